#!/usr/bin/env python
"""Throughput of the OKLS step on one GB300 (or N replicas under torchrun).

Metric: preconditioned matrices per second of okls_step (and dense TFLOP/s)
on the 1.2B-shaped Llama layer set: 24 layers x {q,k,v,o 2048x2048;
gate,up 5504x2048; down 2048x5504} = 168 matrices, bf16 W and G, fp32 state,
Kronecker-structured gradients with condition number 1e3.  One step is one
okls_step call per shape group over all 168 matrices.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl okls|reference]

The JSON line carries the device-resident number (`value`), the end-to-end
number through the public API with pinned host copies (`e2e`), the live
per-launch roofline of the GEMM kernel (`roofline`), the float64 CPU oracle
timed on a bounded sample (`cpu_baseline`) and the SM clocks seen during the
timed region (`clocks`).
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "preconditioned matrices/s per okls_step (TFLOP/s vs GB300 FP16 peak alongside)"
L2_BYTES = 129e6  # GB300 L2
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def dense_flops(m: int, n: int, method: str = "okls") -> float:
    """Dense algorithmic FLOPs of one matrix's step.  OKLS: 27 products of
    each Newton-Schulz chain, the two preconditioned factor inputs and the
    two factor products, the whitening.  Classic Shampoo: two chained chains
    (54 products) per factor, the two factor products of G, the whitening.
    SOAP: three two-sided rotations and the two factor products (the
    eigenbasis refresh is not counted)."""
    if method == "soap":
        return 3 * 2.0 * m * n * (m + n) + 2.0 * m * n * (m + n)
    if method == "shampoo":
        return 54 * 2.0 * (m ** 3 + n ** 3) + 2.0 * m * n * (m + n) + 2.0 * m * n * (m + n)
    return 27 * 2.0 * (m ** 3 + n ** 3) + 4.0 * m * n * (m + n) + 2.0 * m * n * (m + n)


GEMM_SOURCES = ["kronecker_factored_second_gb300/csrc/okls_gemm.cu",
                "kronecker_factored_second_gb300/csrc/okls_epilogue.cuh",
                "kronecker_factored_second_gb300/csrc/okls_ptx.cuh",
                "kronecker_factored_second_gb300/csrc/okls_internal.h"]
TRAFFIC_RECORD = "profiles/okls_gemm_kernel__llama1.2b_dram.json"


def gemm_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def gemm_traffic() -> float | None:
    """DRAM bytes (read + write) per GEMM launch of the headline step, from
    the committed ncu record, or None when the kernel's sources changed since
    those counters were taken."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_RECORD)) as fh:
            rec = json.load(fh)
        if rec.get("source_sha256") != gemm_sources_sha256():
            return None
        return float(rec["traffic_bytes_per_launch"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[2]))
            except ValueError:
                pass
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w": statistics.median(pw) if pw else None, "reasons": sorted(reasons)}


# ------------------------------------------------------------- distributed
def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_setup(ws: int, backend: str):
    if ws > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    """Largest value over ranks (the job's time is its slowest rank's)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------ CPU baseline
def _oracle_threads() -> int:
    return int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1)))


class OracleShapes:
    """The float64 oracle as it stands, one matrix per distinct shape of the
    workload, each with its own state carried from step to step.  A step of
    the whole workload is extrapolated as sum over shapes of (matrices of
    that shape) x (time of one oracle step on that shape): the oracle's cost
    is that of its eigendecompositions and products, which do not depend on
    the values, so iid N(0, 1) gradients of the same shapes stand in."""

    def __init__(self, wl, seed: int = 7):
        import numpy as np

        import oracle as O
        self.O = O
        self.np = np
        self.rng = np.random.default_rng(seed)
        self.hp = O.Hyper(ridge=1e-3)
        self.shapes = []
        for g in wl.groups:
            m, n = g.m, g.n
            st = O.init_state(m, n, self.hp)
            W = self.rng.standard_normal((m, n)) * 1e-3
            self.shapes.append([g, st, W])
        self.matrices = wl.matrices

    def step(self) -> tuple[float, list]:
        """One oracle step per shape; returns the extrapolated seconds of one
        step of the whole workload and the per-shape seconds."""
        per = []
        total = 0.0
        for item in self.shapes:
            g, st, W = item
            G = self.rng.standard_normal((g.m, g.n))
            t0 = time.perf_counter()
            st, W, _U = self.O.okls_step(st, W, G, self.hp.lr, self.hp)
            dt = time.perf_counter() - t0
            item[1], item[2] = st, W
            per.append(dt)
            total += g.batch * dt
        return total, per

    def describe(self, per: list) -> str:
        return ("extrapolation: one float64 oracle step (eigendecomposition roots) per distinct shape, "
                + ", ".join(f"{g.m}x{g.n} {dt:.2f} s x {g.batch}" for (g, _s, _W), dt in zip(self.shapes, per))
                + f" = {sum(g.batch * dt for (g, _s, _W), dt in zip(self.shapes, per)):.1f} s per step of "
                  f"{self.matrices} matrices (iid N(0,1) gradients of the same shapes)")


def oracle_sample(wl) -> dict:
    """cpu_baseline: one oracle step per distinct shape, extrapolated to the
    workload's step (about 10-20 s of host CPU work on the 1.2B-shaped set)."""
    orc = OracleShapes(wl)
    total, per = orc.step()
    return {"value": orc.matrices / total, "unit": "matrices/s", "cores": _oracle_threads(), "kind": "oracle",
            "sample": orc.describe(per)}


def run_reference(args):
    """`--impl reference`: the float64 CPU oracle timed on the host cores,
    each step one oracle step per distinct shape of the workload,
    extrapolated to the whole step (OracleShapes)."""
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    from kronecker_factored_second_gb300.workloads import workload
    wl = workload(args.workload, layers=args.layers)
    orc = OracleShapes(wl, seed=11)
    for _ in range(args.warmup):
        orc.step()
    tot, pers = 0.0, []
    for _ in range(args.steps):
        t, per = orc.step()
        tot += t
        pers.append(per)
    dt = tot / max(args.steps, 1)
    per_mean = [sum(p[i] for p in pers) / len(pers) for i in range(len(orc.shapes))]
    v = orc.matrices / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "matrices/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(wl)},
            "cpu_baseline": {"value": v, "unit": "matrices/s", "cores": _oracle_threads(), "kind": "oracle",
                             "sample": orc.describe(per_mean)},
            "e2e": {"value": v, "unit": "matrices/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_desc(wl) -> str:
    return (f"{wl.name}: " + ", ".join(f"{g.batch} x {g.m}x{g.n} {g.name}" for g in wl.groups)
            + f" = {wl.matrices} matrices, {wl.groups[0].dtype} W and G, fp32 state, "
            f"{wl.recipe} gradients (condition number {wl.cond:g})")


# --------------------------------------------------------------- GPU arm
def run_okls(args):
    import torch

    from kronecker_factored_second_gb300.okls import OklsBatch
    from kronecker_factored_second_gb300.workloads import GradientStream, workload

    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_setup(ws, "nccl")
    wl = workload(args.workload, layers=args.layers)
    # every rank owns a full layer set of its own (weak scaling): seeds differ
    wl.seed = wl.seed + 1000 * rank
    gs = GradientStream(wl, dev)
    n_distinct = max(2, min(wl.steps, args.distinct))
    groups = []
    extra = {}
    if args.method == "soap":
        # SOAP's Adam hyperparameters; the eigenbases are refreshed every 10 steps
        extra = dict(beta1=0.95, beta2=0.95, eps=1e-8, weight_decay=0.0, root_every=args.root_every)
    for gi, g in enumerate(wl.groups):
        ob = OklsBatch(g.batch, g.m, g.n, param_dtype=g.dtype, ns_split_iters=args.split, ridge=args.ridge,
                       method=args.method, device=dev, **extra)
        W = gs.init_weights(gi)
        Gs = [gs.grad(gi, t + 1) for t in range(n_distinct)]
        groups.append((g, ob, W, Gs))
    del gs
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    matrices = wl.matrices
    flops_step = sum(g.batch * dense_flops(g.m, g.n, args.method) for g in wl.groups)
    in_bytes = sum(G[0].numel() * G[0].element_size() for (_g, _ob, _W, G) in groups)
    state_bytes = sum(ob.state.numel() for (_g, ob, _W, _G) in groups)

    def one_step(k):
        for (g, ob, W, Gs) in groups:
            ob.step(W, Gs[k % len(Gs)], args.lr)

    for k in range(args.warmup):
        one_step(k)
    torch.cuda.synchronize()
    for (_g, ob, _W, _G) in groups:
        st = ob.status_nothrow()
        if st[1]:
            raise RuntimeError(f"device status 0x{st[1]:x} during warm-up")
        ob.read_profile()
        ob.profile(True)

    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(dev).uuid)
        if not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        gpu_uuid = None
    clocks = ClockSampler(gpu_uuid) if rank == 0 else None
    barrier(ws)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.5)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(args.steps):
        one_step(args.warmup + k)
    e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    barrier(ws)
    ms_total = e0.elapsed_time(e1)
    ms_total = max_over_ranks(ms_total, ws, dev)
    prof = {"kernel_launches": 0, "gemm_launches": 0, "gemm_flops": 0.0, "gemm_ms": 0.0, "ns_flops": 0.0,
            "ns_ms": 0.0, "ns_launches": 0, "bw_launches": 0, "bw_bytes": 0.0, "bw_ms": 0.0}
    for (_g, ob, _W, _G) in groups:
        p = ob.read_profile()
        for k in prof:
            prof[k] += p[k]
        ob.profile(False)
        st = ob.status_nothrow()
        if st[1]:
            raise RuntimeError(f"device status 0x{st[1]:x} in the timed region")
    ms_step = ms_total / args.steps
    total_matrices = sum_over_ranks(matrices * args.steps, ws, dev)
    value = total_matrices / (ms_total / 1e3)
    tflops = sum_over_ranks(flops_step * args.steps, ws, dev) / (ms_total / 1e3) / 1e12

    peaks, peak_kind = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    achieved = prof["gemm_flops"] / (prof["gemm_ms"] / 1e3) / 1e12 if prof["gemm_ms"] > 0 else None
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    bw_gbs = prof["bw_bytes"] / (prof["bw_ms"] / 1e3) / 1e9 if prof["bw_ms"] > 0 else None
    elementwise = {"kernels": "k_momentum_stats, k_pack, k_normalise (k_sumsq in Shampoo mode)",
                   "bound": "hbm", "achieved": bw_gbs, "peak": hbm, "unit": "GB/s",
                   "frac": (bw_gbs / hbm) if bw_gbs else None,
                   "bytes_per_step": prof["bw_bytes"] / args.steps, "launches_per_step": prof["bw_launches"] / args.steps,
                   "ms_per_step": prof["bw_ms"] / args.steps,
                   "share_of_step": prof["bw_ms"] / ms_total if ms_total > 0 else None,
                   "peak_kind": f"{peak_kind} copy bandwidth"}
    ns_achieved = prof["ns_flops"] / (prof["ns_ms"] / 1e3) / 1e12 if prof["ns_ms"] > 0 else None

    # ---------------------------------------------- end to end (host buffers)
    # Every step copies that step's gradients from pinned host memory and
    # reads the updated parameters back.  The copies run on their own stream
    # and overlap the other shape groups' steps, as a training loop would:
    # group i's step waits for its gradient copy, and its W read-back runs
    # while group i+1 computes.  The timed region starts before the first
    # copy and ends after the last read-back (both events on the copy stream).
    e2e = None
    if not args.no_e2e:
        hostG = []
        for (g, ob, W, Gs) in groups:
            hostG.append([Gs[i].cpu().pin_memory() for i in range(2)])
        devG = [[torch.empty_like(Gs[0]) for _ in range(2)] for (_g, _ob, _W, Gs) in groups]
        hostW = [torch.empty(W.shape, dtype=W.dtype, pin_memory=True) for (_g, _ob, W, _G) in groups]
        h2d = sum(h[0].numel() * h[0].element_size() for h in hostG)
        d2h = sum(h.numel() * h.element_size() for h in hostW)
        copy = torch.cuda.Stream(device=dev)
        ng = len(groups)
        g_ready = [[torch.cuda.Event() for _ in range(2)] for _ in range(ng)]
        w_done = [torch.cuda.Event() for _ in range(ng)]
        w_read = [torch.cuda.Event() for _ in range(ng)]

        def e2e_steps(k0, count):
            # prefetch the first step's gradients
            with torch.cuda.stream(copy):
                for i in range(ng):
                    devG[i][k0 % 2].copy_(hostG[i][k0 % 2], non_blocking=True)
                    g_ready[i][k0 % 2].record(copy)
            for k in range(k0, k0 + count):
                buf = k % 2
                for i, (g, ob, W, _Gs) in enumerate(groups):
                    stream.wait_event(g_ready[i][buf])
                    if k > k0:
                        stream.wait_event(w_read[i])   # W must be read back before it changes again
                    ob.step(W, devG[i][buf], args.lr)
                    w_done[i].record(stream)
                    with torch.cuda.stream(copy):
                        copy.wait_event(w_done[i])
                        hostW[i].copy_(W, non_blocking=True)
                        w_read[i].record(copy)
                        if k + 1 < k0 + count:
                            # next step's gradients into the other buffer (its last reader
                            # was this group's previous step, finished before w_done)
                            devG[i][1 - buf].copy_(hostG[i][(k + 1) % 2], non_blocking=True)
                            g_ready[i][1 - buf].record(copy)

        e2e_steps(0, max(1, args.warmup // 2))
        torch.cuda.synchronize()
        barrier(ws)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(copy)
        stream.wait_event(a)
        e2e_steps(0, args.steps)
        copy.wait_stream(stream)
        b.record(copy)
        torch.cuda.synchronize()
        barrier(ws)
        ms_e2e = max_over_ranks(a.elapsed_time(b), ws, dev)
        e2e = {"value": sum_over_ranks(matrices * args.steps, ws, dev) / (ms_e2e / 1e3), "unit": "matrices/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e / args.steps,
               "copies": "pinned host, own stream, overlapped with the other groups' steps"}
        del hostG, devG, hostW

    # --------------------------------- other modes, timed the same way
    def rebuild(**kw):
        torch.cuda.synchronize()
        for i in range(len(groups)):
            g, ob, W, Gs = groups[i]
            ob.close()
            groups[i] = (g, None, W, Gs)
            del ob
            torch.cuda.empty_cache()
            groups[i] = (g, OklsBatch(g.batch, g.m, g.n, param_dtype=g.dtype, device=dev, **kw), W, Gs)

    def timed():
        for k in range(args.warmup):
            one_step(k)
        torch.cuda.synchronize()
        for (_g, ob, _W, _G) in groups:
            st = ob.status_nothrow()
            if st[1]:
                raise RuntimeError(f"device status 0x{st[1]:x} during warm-up")
            ob.read_profile()
            ob.profile(True)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in range(args.steps):
            one_step(k)
        b.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(a.elapsed_time(b), ws, dev)
        gf, gm = 0.0, 0.0
        for (_g, ob, _W, _G) in groups:
            p = ob.read_profile()
            gf += p["gemm_flops"]
            gm += p["gemm_ms"]
            st = ob.status_nothrow()
            if st[1]:
                raise RuntimeError(f"device status 0x{st[1]:x} in the timed region")
        return ms, (gf / (gm / 1e3) / 1e12 if gm > 0 else None)

    split_line = None
    if args.also_split and args.split == 0 and args.method == "okls":
        rebuild(ns_split_iters=3, ridge=1e-4)
        ms2, gt = timed()
        split_line = {"mode": "iterations 0-2 split (hi/lo binary16), ridge 1e-4, 41 NS products per factor",
                      "value": sum_over_ranks(matrices * args.steps, ws, dev) / (ms2 / 1e3),
                      "unit": "matrices/s", "ms_per_step": ms2 / args.steps,
                      "tflops_dense_27": sum_over_ranks(flops_step * args.steps, ws, dev) / (ms2 / 1e3) / 1e12,
                      "gemm_tflops_executed": gt}
    plain_line = None
    if args.also_plain and args.split == 0 and args.method == "okls":
        rebuild(ns_split_iters=10, ridge=0.0)
        ms6, gt = timed()
        plain_line = {"mode": "every iteration split (hi/lo binary16), no ridge: the root of the unridged factor "
                              "(81 binary16 products per factor)",
                      "value": sum_over_ranks(matrices * args.steps, ws, dev) / (ms6 / 1e3),
                      "unit": "matrices/s", "ms_per_step": ms6 / args.steps,
                      "tflops_dense_27": sum_over_ranks(flops_step * args.steps, ws, dev) / (ms6 / 1e3) / 1e12,
                      "gemm_tflops_executed": gt}
    shampoo_line = None
    if args.also_shampoo and args.method == "okls":
        rebuild(ridge=args.ridge, method="shampoo", lr=args.lr, weight_decay=0.0)
        ms3, gt = timed()
        fs = sum(g.batch * dense_flops(g.m, g.n, "shampoo") for g in wl.groups)
        shampoo_line = {"method": "classic Shampoo: summed factors, L^-1/4 G R^-1/4 by two chained "
                                  "Newton-Schulz runs (54 binary16 products per factor), ridge "
                                  f"{args.ridge:g}, roots every step",
                        "value": sum_over_ranks(matrices * args.steps, ws, dev) / (ms3 / 1e3),
                        "unit": "matrices/s", "ms_per_step": ms3 / args.steps,
                        "tflops_dense": sum_over_ranks(fs * args.steps, ws, dev) / (ms3 / 1e3) / 1e12,
                        "gemm_tflops": gt}

    clean_large_line = None
    if args.also_clean_large and args.method == "okls" and args.workload == "llama1.2b":
        # Clean over the same layer set with the pages' 1.3B settings: rank 256,
        # oversampling 8, one power iteration, a refresh every 10 steps, betas 0.95
        rebuild(method="clean", rank=256, oversample=8, power_iters=1, root_every=10, beta1=0.95, beta2=0.95,
                eps=1e-8, weight_decay=0.0, lr=args.lr)
        cgen = torch.Generator(device=dev)
        cgen.manual_seed(wl.seed + 29)
        cnoise = [torch.randn(ob.noise_shape, generator=cgen, device=dev) for (_g, ob, _W, _G) in groups]

        def clean_step(k):
            for i, (_g, ob, W, Gs) in enumerate(groups):
                ob.step(W, Gs[k % len(Gs)], args.lr, noise=cnoise[i] if ob.refresh_due else None)
        for k in range(3):
            clean_step(k)
        torch.cuda.synchronize()
        csteps = 20
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in range(csteps):
            clean_step(k)
        b.record(stream)
        torch.cuda.synchronize()
        for (_g, ob, _W, _G) in groups:
            if ob.status_nothrow()[1]:
                raise RuntimeError("device status flagged in the Clean leg")
        ms5 = max_over_ranks(a.elapsed_time(b), ws, dev)
        clean_large_line = {
            "method": "Clean (block Adam in rank-256 Nystrom bases, oversampling 8, one power iteration, refresh "
                      "every 10 steps, betas 0.95); batched fp32 GEMMs, k x k work in one CTA per matrix",
            "workload": "the same 168-matrix layer set, bf16 W and G", "steps": csteps,
            "value": sum_over_ranks(matrices * csteps, ws, dev) / (ms5 / 1e3), "unit": "matrices/s",
            "ms_per_step": ms5 / csteps,
            "state_gb": sum(ob.state.numel() for (_g, ob, _W, _G) in groups) / 1e9}
        del cnoise

    soap_large_line = None
    if args.also_soap_large and args.method == "okls" and args.workload == "llama1.2b":
        # SOAP over the same layer set (betas 0.95, refresh every 10 steps): the
        # warm-up holds the first refresh (from the identity), the timed steps
        # one refresh warm-started from the previous bases
        try:
            rebuild(method="soap", root_every=10, beta1=0.95, beta2=0.95, eps=1e-8, weight_decay=0.0, lr=args.lr)

            def soap_step(k):
                for (_g, ob, W, Gs) in groups:
                    ob.step(W, Gs[k % len(Gs)], args.lr)
            for k in range(10):
                soap_step(k)
            torch.cuda.synchronize()
            ssteps = 10
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for k in range(ssteps):
                soap_step(10 + k)
            b.record(stream)
            torch.cuda.synchronize()
            for (_g, ob, _W, _G) in groups:
                if ob.status_nothrow()[1]:
                    raise RuntimeError("device status flagged in the SOAP leg")
            ms6 = max_over_ranks(a.elapsed_time(b), ws, dev)
            fs = sum(g.batch * dense_flops(g.m, g.n, "soap") for g in wl.groups)
            soap_large_line = {
                "method": "SOAP (Adam in the factors' eigenbases, refresh every 10 steps, betas 0.95); "
                          "fp32-accurate products on the tensor cores (three-term bf16 split), blocked Jacobi "
                          "refresh", "workload": "the same 168-matrix layer set, bf16 W and G, fp32 state",
                "steps": ssteps, "warmup": 10,
                "value": sum_over_ranks(matrices * ssteps, ws, dev) / (ms6 / 1e3), "unit": "matrices/s",
                "ms_per_step": ms6 / ssteps,
                "tflops_products": sum_over_ranks(fs * ssteps, ws, dev) / (ms6 / 1e3) / 1e12,
                "state_gb": sum(ob.state.numel() for (_g, ob, _W, _G) in groups) / 1e9}
        except Exception as e:  # the headline line is printed either way
            soap_large_line = {"error": str(e)[:300]}

    def small_leg(method, wl_name="single128x64", nsteps=200, **kw):
        """A small workload for the SOAP and Clean modes (one 128 x 64 matrix
        by default), `nsteps` timed steps after 20 warm-up steps; Clean's
        Gaussian draws are drawn up front and stay resident like the
        gradients."""
        swl = workload(wl_name)
        sgs = GradientStream(swl, dev)
        sg = swl.groups[0]
        sob = OklsBatch(sg.batch, sg.m, sg.n, param_dtype=sg.dtype, method=method, beta1=0.95, beta2=0.95,
                        eps=1e-8, weight_decay=0.0, root_every=10, device=dev, **kw)
        sW = sgs.init_weights(0)
        sG = [sgs.grad(0, t + 1) for t in range(4)]
        gen = torch.Generator(device=dev)
        gen.manual_seed(swl.seed + 17)
        noise = [torch.randn(sob.noise_shape, generator=gen, device=dev) for _ in range(4)] \
            if method == "clean" else None

        def st(k):
            sob.step(sW, sG[k % 4], 3e-3, noise=noise[k % 4] if noise and sob.refresh_due else None)
        for k in range(20):
            st(k)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for k in range(nsteps):
            st(k)
        b.record(stream)
        torch.cuda.synchronize()
        if sob.status_nothrow()[1]:
            raise RuntimeError(f"device status flagged in the {method} leg")
        ms4 = a.elapsed_time(b)
        sob.close()
        desc = {"single128x64": "single128x64: one 128 x 64 fp32 matrix",
                "batch16x512": "batch16x512: 16 x 512 x 512 fp32 matrices"}[wl_name]
        return {"workload": desc, "steps": nsteps,
                "value": sg.batch * nsteps / (ms4 / 1e3), "unit": "matrices/s", "ms_per_step": ms4 / nsteps}

    soap_line = clean_line = None
    if args.also_soap and args.method == "okls":
        soap_line = {"method": "SOAP (Adam in the factors' eigenbasis), fp32, one CTA per matrix, Jacobi refresh "
                               "every 10 steps", **small_leg("soap")}
    soap512_line = clean512_line = None
    if args.also_soap and args.method == "okls":
        soap512_line = {"method": "SOAP as above on the batched-GEMM path (Jacobi eigensolves with logged rotations, "
                                  "the matrix in L2 at d = 512), refresh every 10 steps", **small_leg("soap", "batch16x512", 50)}
    if args.also_clean and args.method == "okls":
        clean512_line = {"method": "Clean, rank 56 + oversampling 8, one power iteration, refresh every 10 steps, "
                                   "batched-GEMM path",
                         **small_leg("clean", "batch16x512", 50, rank=56, oversample=8, power_iters=1)}
    if args.also_clean and args.method == "okls":
        clean_line = {"method": "Clean (block Adam in rank-16 Nystrom bases, oversampling 8, one power iteration), "
                                "fp32, one CTA per factor, refresh every 10 steps",
                      **small_leg("clean", rank=16, oversample=8, power_iters=1)}

    cpu = None
    if rank == 0 and ws >= 1 and not args.no_cpu_baseline:
        cpu = oracle_sample(wl)

    if rank == 0:
        # SOAP's products run on other kernels than the per-launch events
        # time: no roofline object for that mode
        roofline = None if args.method == "soap" else {
            "bound": "tensor", "kernel": "okls_gemm_kernel (tcgen05, all products of the step)",
            "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
            "frac": (achieved / peak) if achieved else None, "traffic": gemm_traffic(),
            "traffic_unit": "bytes per launch (dram read + write, ncu, full-size step)",
            "peak_kind": f"{peak_kind} bf16 sustained (fp16 nominal ratio 1)",
            "launches": prof["gemm_launches"], "ms_per_launch": prof["gemm_ms"] / max(1, prof["gemm_launches"]),
            "ns_chain_tflops": ns_achieved,
            "ns_chain_frac": (ns_achieved / peak) if ns_achieved else None}
        line = {
            "metric": METRIC, "value": value, "unit": "matrices/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp32" if args.method == "soap" else "fp16", "data": "synthetic",
            "config": {
                "workload": workload_desc(wl),
                "method": args.method,
                "precision": ("fp32-accurate throughout (products on the tensor cores as three-term bf16 splits "
                              "with fp32 accumulation; blocked Jacobi eigenbasis refresh every "
                              f"{args.root_every} steps)" if args.method == "soap" else
                              f"binary16 Newton-Schulz operands, fp32 accumulation, split_iters={args.split}, "
                              f"ridge={args.ridge:g}"),
                "l2": (f"inputs larger than L2: {in_bytes / 1e9:.2f} GB of gradients and "
                       f"{state_bytes / 1e9:.1f} GB of state per step"
                       if in_bytes + state_bytes > L2_BYTES else
                       f"inputs and state fit in L2 ({(in_bytes + state_bytes) / 1e6:.0f} MB); L2 not flushed "
                       f"between steps"),
                "parallelism": f"owner-computes replicas x{ws} (each rank a full layer set)"},
            "tflops": tflops,
            "tflops_frac_of_peak": tflops / peak,
            "roofline": roofline,
            "elementwise": elementwise,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": prof["kernel_launches"],
            "clocks": clk,
        }
        if split_line:
            line["split_mode"] = split_line
        if plain_line:
            line["plain_root_mode"] = plain_line
        if shampoo_line:
            line["shampoo"] = shampoo_line
        if soap_line:
            line["soap"] = soap_line
        if clean_line:
            line["clean"] = clean_line
        if clean_large_line:
            line["clean_large"] = clean_large_line
        if soap_large_line:
            line["soap_large"] = soap_large_line
        if soap512_line:
            line["soap_512"] = soap512_line
        if clean512_line:
            line["clean_512"] = clean512_line
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["okls", "reference"], default="okls")
    ap.add_argument("--workload", default="llama1.2b")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count (small profiling cases)")
    ap.add_argument("--split", type=int, default=0)
    ap.add_argument("--ridge", type=float, default=1e-3)
    ap.add_argument("--lr", type=float, default=0.09434)
    ap.add_argument("--distinct", type=int, default=4, help="distinct gradient batches kept on the device")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--also-split", type=int, default=1)
    ap.add_argument("--also-plain", type=int, default=1)
    ap.add_argument("--also-shampoo", type=int, default=1)
    ap.add_argument("--also-soap", type=int, default=1)
    ap.add_argument("--also-clean", type=int, default=1)
    ap.add_argument("--also-clean-large", type=int, default=1)
    ap.add_argument("--also-soap-large", type=int, default=1)
    ap.add_argument("--method", choices=["okls", "shampoo", "soap"], default="okls")
    ap.add_argument("--root-every", type=int, default=10, help="SOAP: eigenbasis refresh interval")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "okls":
        print("note: at least 3 warm-up steps are used", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_okls(args)


if __name__ == "__main__":
    main()
