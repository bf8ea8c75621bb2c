"""Benchmark: the block-quantized weight matmul on one GB300, over the five seeded synthetic workloads.

A step is one pass of the whole hot path over the workload the pages time (candle PR 4056, "Metal:
64-token tile for the quantized matrix-matrix kernel", section "This branch, kernel level"): the seven
projections of one Qwen3-Embedding-4B layer (attn_q/k/v/output Q4_K/Q6_K, ffn_gate/up Q4_K, ffn_down Q6_K)
at every token count M in {1, 2, 7, 32, 33, 64, 96, 100, 128, 130, 136, 512, 2048}, plus the 65-token case
as a batch of two sequences: 105 projections. M <= 16 runs the mat-vec path, larger M the tcgen05 path. At
M <= 16 the projections that share an input and a type go in one qmm_batch launch (attn_q + attn_k,
ffn_gate + ffn_up), as a model chains them; the `unbatched` object times every projection as its own call.
All calls pass QMM_W_STATIC (the weights are model data that no kernel of the step writes).

Metric: weight-GB/s of the M <= 16 calls against HBM (value), and TFLOPS of the M >= 64 calls against the
bf16 tensor-core peak (tflops_m_ge_64). Inputs are resident in HBM; weights rotate through 7 copies of the
layer (447 MB, more than 3x the 129 MB L2) so that no call reads weights another call left in L2.

Roofline (per call): t_roof = max((weight + activation bytes) / HBM copy peak, 2 M N K / bf16 burst peak);
a set of calls is at sum(t_roof) / sum(t_measured). Reported per class (M <= 16, 17..136, >= 512), for the
whole step, and for the dominant kernel (the class that takes the most time).

The other workloads are timed in the same run and reported as objects of the same JSON line: the small
Q4_0 matrix at 1 and 7 tokens (small_q4_0), the Qwen3-0.6B-shaped decode layer with group-64 affine 4-bit
weights (qwen3_06b), the expert-indexed product (moe) and the all-type sweep (sweep).
The e2e figure times the M <= 16 calls through the C-ABI with activations copied from pinned host memory and
results copied back inside the timed region.

    python bench.py [--steps K] [--warmup W] [--gpus N] [--impl ours|reference] [--case NAME:M | moe:N]
                    [--no-cpu] [--no-moe] [--no-extra] [--detail]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthetic  # noqa: E402

METRIC = "qmatmul weight-GB/s vs HBM peak (M≤16); TFLOPS vs bf16 MMA peak (M≥64)"
LAYER = synthetic.QWEN3_EMB_4B_LAYER
TOKENS = synthetic.QWEN3_EMB_4B_TOKENS
BATCH2 = synthetic.QWEN3_EMB_4B_BATCH2_TOKENS
COPIES = 7
BPW = {"Q4_K": 4.5, "Q6_K": 6.5625}
WORKLOAD = ("Qwen3-Embedding-4B layer: attn_q 4096x2560 Q4_K, attn_k 1024x2560 Q4_K, attn_v 1024x2560 Q6_K, "
            "attn_output 2560x4096 Q4_K, ffn_gate/ffn_up 9728x2560 Q4_K, ffn_down 2560x9728 Q6_K; "
            "M in {1,2,7,32,33,64,96,100,128,130,136,512,2048} + 2x65; fp32 activations N(0,1), "
            "weights N(0,0.02) quantized")


# DRAM traffic of the dominant call class, from one ncu capture of the bench's own step
# (dram__bytes_read.sum + dram__bytes_write.sum of every launch, attributed to the calls in launch order;
# one pass): bytes per call over all the class's launches (the tensor-core kernel and its helper kernels),
# with the algorithmic bytes per call (weights + binary32 activations) and launches per call beside it.
# Valid only for the kernel and planner sources it was taken on: None once one of them has changed.
TRAFFIC = {"class": "m_17_136", "bytes_per_call": 16.160e6, "algorithmic_bytes_per_call": 10.415e6,
           "launches_per_call": 2.8, "mm_kernel_bytes_per_call": 9.840e6,
           "sources": ["weight_quantized_matmul_fly_gb300/csrc/k_mm.cu", "weight_quantized_matmul_fly_gb300/csrc/mm_slab.cuh",
                       "weight_quantized_matmul_fly_gb300/csrc/ptx.cuh", "weight_quantized_matmul_fly_gb300/csrc/qmm_abi.cu"],
           "sha256": "c4eaf06286c178678fc58a22160d24c8241cbd7ce1a9d3fbcf1a6a185084e4fb"}


def sources_digest(paths):
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(cls):
    """The recorded DRAM traffic of this call class, or None (not measured on these sources)."""
    if TRAFFIC["class"] != cls or not TRAFFIC["sha256"]:
        return None
    try:
        if sources_digest(TRAFFIC["sources"]) != TRAFFIC["sha256"]:
            return None
    except OSError:
        return None
    return {k: TRAFFIC[k] for k in ("bytes_per_call", "algorithmic_bytes_per_call", "launches_per_call",
                                    "mm_kernel_bytes_per_call")}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# Projections that take the same input and share a type: at M <= 16 a step serves each pair with one
# qmm_batch launch, as a model chains them (the query and key projections of the attention input; the gate
# and up projections of the feed-forward input). attn_v shares the input but not the type (Q6_K).
SHARED_INPUT = {"attn_q": "attn_k", "ffn_gate": "ffn_up"}
SHARED_PARTNERS = set(SHARED_INPUT.values())


def bench_config(world):
    """The workload of a step, the same dict on both arms."""
    return {"workload": WORKLOAD, "calls_per_step": len(calls_of_step()),
            "l2": "rotating %d weight copies (%.0f MB), inputs larger than L2" % (
                COPIES, COPIES * sum(weight_bytes(N, K, qt) for _, N, K, qt in LAYER) / 1e6),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def calls_of_step():
    """(name, N, K, qtype, M, batch_index) for one step, grouped by M so consecutive calls touch
    different matrices."""
    out = []
    for M in TOKENS:
        for name, N, K, qt in LAYER:
            out.append((name, N, K, qt, M, 0))
        if M == 64:  # the 65-token batch of two sits between 64 and 96 in token order
            for b in range(2):
                for name, N, K, qt in LAYER:
                    out.append((name, N, K, qt, BATCH2, b))
    return out


def weight_bytes(N, K, qt):
    return N * K * BPW[qt] / 8


class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", "qmm_clocks_%d.csv" % os.getpid())

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if not self.proc or not os.path.exists(self.path):
            return None
        sm, smax, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [s.strip() for s in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = max(smax, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def max_over_ranks(pg, v, device=None):
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def whole_job(pg, units_per_rank, seconds, world, device=None):
    """Whole-job throughput of N replicas doing the same work: the units all ranks processed divided by the
    slowest rank's time."""
    return units_per_rank * world / max_over_ranks(pg, seconds, device)


def call_roofline(M, N, K, wbytes, x_elem_bytes, peaks):
    """(roofline time in us, bound) of one call: max(bytes / HBM, flops / bf16 burst peak)."""
    t_hbm = (wbytes + M * K * x_elem_bytes) / (peaks["hbm_gbs"] * 1e9) * 1e6
    t_mma = 2.0 * M * N * K / (peaks["bf16_tflops"] * 1e12) * 1e6
    return (t_hbm, "hbm") if t_hbm >= t_mma else (t_mma, "tensor")


def class_summary(idx, calls, call_ms, rf, peaks):
    t_meas = sum(call_ms[i] for i in idx) * 1e3
    t_roof = sum(rf[i][0] for i in idx)
    t_hbm = sum(rf[i][0] for i in idx if rf[i][1] == "hbm")
    wb = sum(weight_bytes(calls[i][1], calls[i][2], calls[i][3]) for i in idx)
    fl = sum(2.0 * calls[i][4] * calls[i][1] * calls[i][2] for i in idx)
    return {"calls": len(idx), "us_measured": round(t_meas, 2), "us_roofline": round(t_roof, 2),
            "frac": round(t_roof / t_meas, 4), "bound": "hbm" if t_hbm >= 0.5 * t_roof else "tensor",
            "weight_gbs": round(wb / t_meas / 1e3, 1), "tflops": round(fl / t_meas / 1e6, 2)}


# ---------------------------------------------------------------------------------------- our arm

def run_ours(args):
    import torch
    import weight_quantized_matmul_fly_gb300 as qmm

    world, rank, local, pg = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    qmm.build()
    peaks = load_peaks()

    if args.case and args.case.startswith("moe:"):
        if rank == 0:
            run_moe_case(args, qmm, torch, dev, peaks, int(args.case.split(":")[1]))
        if pg:
            pg.destroy_process_group()
        return
    calls = calls_of_step()
    if args.case:
        name, m = args.case.split(":")
        calls = [c for c in calls if c[0] == name and c[4] == int(m) and c[5] == 0]
        assert calls, "no such case"

    # weights: 7 copies of the layer, quantized on the device from seeded binary32 weights
    wq = {}
    for copy in range(COPIES):
        for name, N, K, qt in LAYER:
            w32 = torch.from_numpy(synthetic.weights(N, K, seed=copy)).to(dev)
            buf = torch.empty(qmm.row_bytes(qt, K) * N, dtype=torch.uint8, device=dev)
            qmm.qmm_quantize(w32, qt, N, K, buf)
            wq[(copy, name)] = buf
            del w32
    xs, ys, ys2 = {}, {}, {}
    ws_bytes = 0
    for name, N, K, qt, M, b in calls:
        if (M, K, b) not in xs:
            xs[(M, K, b)] = torch.from_numpy(synthetic.activations(M, K, seed=M + 17 * b)).to(dev)
        if (M, N) not in ys:
            ys[(M, N)] = torch.empty((M, N), dtype=torch.float32, device=dev)
            ys2[(M, N)] = torch.empty((M, N), dtype=torch.float32, device=dev)   # a batch partner's output
        ws_bytes = max(ws_bytes, qmm.qmm_workspace_size(qt, N, K, M))
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream()
    L = qmm.lib()
    import ctypes
    P = ctypes.c_void_p

    ncalls = len(calls)
    names = {c[0] for c in calls}
    per_step_launches = sum(qmm.qmm_launch_count(c[3], c[1], c[2], c[4]) for c in calls
                            if not (c[4] <= 16 and c[0] in SHARED_PARTNERS and
                                    any(SHARED_INPUT.get(n) == c[0] for n in names)))

    # The calls grouped by token count (the 65-token batch of two is one group); inside a captured graph
    # consecutive kernels overlap through programmatic dependent launch.
    groups = []                                   # list of (label, [call indices])
    for i, c in enumerate(calls):
        label = "%dx%d" % (2, c[4]) if c[4] == BATCH2 else str(c[4])
        if not groups or groups[-1][0] != label:
            groups.append((label, []))
        groups[-1][1].append(i)

    def run_group(copy, idxs):
        done = set()
        for i in idxs:
            if i in done:
                continue
            name, N, K, qt, M, b = calls[i]
            partner = SHARED_INPUT.get(name)
            j = next((j for j in idxs if partner and calls[j][0] == partner and calls[j][5] == b), None)
            if M <= 16 and j is not None:
                # the projections that share this input and type: one mat-vec launch (qmm_batch)
                done.add(j)
                N2 = calls[j][1]
                qmm.qmm_batch([wq[(copy, name)], wq[(copy, partner)]], qmm.TYPE_ID[qt] | qmm.W_STATIC, [N, N2], K,
                              xs[(M, K, b)], [ys[(M, N)], ys2[(M, N2)]])
                continue
            rc = L.qmm_ws(P(wq[(copy, name)].data_ptr()), qmm.TYPE_ID[qt] | qmm.W_STATIC, N, K,
                          P(xs[(M, K, b)].data_ptr()), M, P(ys[(M, N)].data_ptr()), P(ws.data_ptr()), ws.numel(),
                          P(stream.cuda_stream))
            if rc:
                raise RuntimeError("qmm_ws: " + qmm.qmm_strerror(rc))

    for s in range(args.warmup):                  # eager warm-up: kernel attributes, occupancy queries
        for _, idxs in groups:
            run_group(s % COPIES, idxs)
    torch.cuda.synchronize()
    # The timed steps: one CUDA graph per weight copy holding the whole step (all groups back to back), the
    # copies replayed in turn. Per-group times: one graph per group holding that group for every weight copy
    # (the layer at that token count seven times over, as a model runs its layers), replayed in steady state;
    # they give the per-token-count figures and the roofline classes.
    graphs, ggraphs = {}, {}
    with torch.cuda.stream(stream):
        for copy in range(COPIES):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _, idxs in groups:
                    run_group(copy, idxs)
            graphs[copy] = g
        for gi, (_, idxs) in enumerate(groups):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for copy in range(COPIES):
                    run_group(copy, idxs)
            ggraphs[gi] = g
    torch.cuda.synchronize()
    for s in range(args.warmup):                  # warm-up replays
        graphs[s % COPIES].replay()
        for gi in range(len(groups)):
            ggraphs[gi].replay()
    torch.cuda.synchronize()

    ng = len(groups)
    t0e = torch.cuda.Event(enable_timing=True)
    t1e = torch.cuda.Event(enable_timing=True)
    gev = [torch.cuda.Event(enable_timing=True) for _ in range(ng + 1)]
    greps = max(2, args.steps // COPIES)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        with Clocks(local) as clk:
            t0e.record(stream)
            for s in range(args.steps):
                graphs[(args.warmup + s) % COPIES].replay()
            t1e.record(stream)
            for gi in range(ng):
                gev[gi].record(stream)
                for _ in range(greps):
                    ggraphs[gi].replay()
            gev[ng].record(stream)
            torch.cuda.synchronize()
    if pg:
        pg.barrier()
    total_ms = max_over_ranks(pg, t0e.elapsed_time(t1e), dev)
    group_ms = np.array([gev[gi].elapsed_time(gev[gi + 1]) / (greps * COPIES) for gi in range(ng)])
    # per-call times are not measured inside a group; spread each group's time over its calls by weight
    # bytes for the per-call table only (the aggregates below use group times)
    call_ms = np.zeros(ncalls)
    for gi, (_, idxs) in enumerate(groups):
        wbs = np.array([weight_bytes(calls[i][1], calls[i][2], calls[i][3]) for i in idxs])
        for i, wbi in zip(idxs, wbs):
            call_ms[i] = group_ms[gi] * wbi / wbs.sum()

    # aggregates
    small = [i for i, c in enumerate(calls) if c[4] <= 16]
    big = [i for i, c in enumerate(calls) if c[4] >= 64]
    wb_small = sum(weight_bytes(calls[i][1], calls[i][2], calls[i][3]) for i in small)
    t_small = sum(call_ms[i] for i in small) * 1e-3
    fl_big = sum(2.0 * calls[i][4] * calls[i][1] * calls[i][2] for i in big)
    t_big = sum(call_ms[i] for i in big) * 1e-3
    gbs = whole_job(pg, wb_small, t_small, world, dev) / 1e9 if small else None
    tfl = whole_job(pg, fl_big, t_big, world, dev) / 1e12 if big else None

    # roofline per call, summed per class (group times: every group holds one token count, so a class,
    # a set of token counts, is a union of groups and its measured time is exact)
    rf = [call_roofline(c[4], c[1], c[2], weight_bytes(c[1], c[2], c[3]), 4, peaks) for c in calls]
    classes = {"m_le_16": lambda m: m <= 16, "m_17_136": lambda m: 17 <= m <= 136, "m_ge_512": lambda m: m >= 512}
    cls_out = {}
    for name, pred in classes.items():
        idx = [i for i, c in enumerate(calls) if pred(c[4])]
        if not idx:
            continue
        cls_out[name] = class_summary(idx, calls, call_ms, rf, peaks)
    step_summary = class_summary(list(range(ncalls)), calls, call_ms, rf, peaks)
    dom = max(cls_out, key=lambda k: cls_out[k]["us_measured"])
    d = cls_out[dom]
    bound = d["bound"]
    peak = peaks["hbm_gbs"] if bound == "hbm" else peaks["bf16_tflops"]
    roof = {"bound": bound, "achieved": round(d["frac"] * peak, 2), "peak": peak,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": d["frac"],
            "traffic": (recorded_traffic(dom) or {}).get("bytes_per_call"), "traffic_detail": recorded_traffic(dom),
            "class": dom, "kernel": ("gtc::gemv_tc_kernel (mma.sync mat-vec)" if dom == "m_le_16"
                                     else "mm::mm_kernel (tcgen05) with its helper kernels"),
            "peak_kind": ("HBM copy" if bound == "hbm" else "bf16 dense, burst") + ", " + peaks["source"],
            "achieved_kind": "sum of per-call roofline times / measured time, times the peak of the bound "
                             "that holds for most of the class's roofline time",
            "algorithmic_per_call": "max((N*K*bpw/8 + M*K*4) / HBM, 2*M*N*K / bf16 peak)",
            "traffic_unit": "DRAM bytes per call of the class over all its launches (ncu over the bench's step), "
                            "null unless measured on the current kernel and planner sources"}

    per_m = {}
    for i, c in enumerate(calls):
        key = "%dx%d" % (2, c[4]) if c[4] == BATCH2 else str(c[4])
        d = per_m.setdefault(key, {"us": 0.0, "wbytes": 0.0, "flops": 0.0, "roof": 0.0})
        d["us"] += call_ms[i] * 1e3
        d["wbytes"] += weight_bytes(c[1], c[2], c[3])
        d["flops"] += 2.0 * c[4] * c[1] * c[2]
        d["roof"] += rf[i][0]
    for k, d in per_m.items():
        d["weight_gbs"] = round(d["wbytes"] / (d["us"] * 1e-6) / 1e9, 1)
        d["tflops"] = round(d["flops"] / (d["us"] * 1e-6) / 1e12, 2)
        d["frac"] = round(d["roof"] / d["us"], 4)
        d["us"] = round(d["us"], 2)
        del d["wbytes"], d["flops"], d["roof"]

    if args.detail:
        print("step %.2f us (whole-step graphs), sum of steady-state groups %.2f us" % (
            total_ms / args.steps * 1e3, group_ms.sum() * 1e3), file=sys.stderr)
        for gi, (label, idxs) in enumerate(groups):
            wb = sum(weight_bytes(calls[i][1], calls[i][2], calls[i][3]) for i in idxs)
            fl = sum(2.0 * calls[i][4] * calls[i][1] * calls[i][2] for i in idxs)
            print("M=%-6s %2d calls %9.2f us %8.1f GB/s %8.2f TFLOP/s" % (
                label, len(idxs), group_ms[gi] * 1e3, wb / (group_ms[gi] * 1e-3) / 1e9,
                fl / (group_ms[gi] * 1e-3) / 1e12), file=sys.stderr)
    unbatched = run_unbatched(args, qmm, torch, dev, wq, peaks) if not args.case else None
    e2e = run_e2e(args, qmm, torch, dev, calls, wq, ws) if not args.case else None
    del wq, xs, ys, graphs, ggraphs
    torch.cuda.empty_cache()
    extra = not args.case and not args.no_extra
    moe = run_moe(args, qmm, torch, dev, peaks) if (not args.case and not args.no_moe) else None
    small_q4_0 = run_small_q4_0(qmm, torch, dev, peaks) if extra else None
    qwen3_06b = run_qwen3_06b(qmm, torch, dev, peaks) if extra else None
    sweep = run_sweep(qmm, torch, dev, peaks) if extra else None
    cpu = cpu_baseline(args) if (rank == 0 and world == 1 and not args.no_cpu and not args.case) else None

    clocks = clk.summary()
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 1) if gbs else None, "unit": "GB/s",
            "tflops_m_ge_64": {"value": round(tfl, 2) if tfl else None, "unit": "TFLOP/s",
                               "frac_of_bf16_burst": round(tfl / peaks["bf16_tflops"], 4) if tfl else None},
            "value_frac_of_hbm": round(gbs / peaks["hbm_gbs"] / world, 4) if gbs else None,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 (M<=16) + bf16 in / f32 accumulate (M>16)", "data": "synthetic",
            "config": bench_config(world) if not args.case else {"workload": "single call " + args.case},
            "roofline": roof, "roofline_classes": cls_out, "roofline_step": step_summary,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": per_step_launches * args.steps,
            "clocks": clocks, "per_m": per_m, "unbatched": unbatched, "small_q4_0": small_q4_0, "qwen3_06b": qwen3_06b, "moe": moe,
            "sweep": sweep, "peaks": peaks,
        }
        print(json.dumps(line))
    if pg:
        pg.destroy_process_group()


def run_moe_case(args, qmm, torch, dev, peaks, n):
    """One expert-indexed workload alone (--case moe:N): N tokens routed top-8 over 128 experts of
    4096 x 1024 Q4_0 (one bank), each expert path called once eagerly in the order 2, 1, 2 (a profiler takes
    the first launch of a kernel), then both paths timed over 16 replayed calls on 8 rotating id tables."""
    E, Nr, TOPK, K = synthetic.MOE_EXPERTS, synthetic.MOE_ROWS, synthetic.MOE_TOPK, 1024
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    rb = qmm.row_bytes("Q4_0", K)
    bank = []
    for _ in range(E):
        w = torch.randn(Nr, K, device=dev, generator=gen) * 0.02
        b = torch.empty(rb * Nr, dtype=torch.uint8, device=dev)
        qmm.qmm_quantize(w, "Q4_0", Nr, K, b)
        bank.append(b)
    idss = [torch.from_numpy(synthetic.expert_ids(n, batch=b)).to(dev) for b in range(8)]
    x = torch.randn(n, K, device=dev, generator=gen)
    y = torch.empty(n, TOPK, Nr, device=dev)
    for path in (2, 1, 2):
        qmm.qmm_id(bank, "Q4_0", Nr, K, x, idss[0], y, path=path)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    row = {"workload": "moe %d tokens, top-8 of 128 experts 4096x1024 Q4_0" % n,
           "auto_path": qmm.qmm_id_pick_path("Q4_0", E, K, n, TOPK)}
    for path in (1, 2):
        fns = [(lambda i=i, path=path: qmm.qmm_id(bank, "Q4_0", Nr, K, x, idss[i % 8], y, path=path))
               for i in range(16)]
        us = time_graph(torch, stream, fns)
        row["us_path%d" % path] = round(us, 2)
        row["tflops_path%d" % path] = round(2.0 * n * TOPK * Nr * K / us / 1e6, 2)
    print(json.dumps(row))


def time_graph(torch, stream, calls, replays=4):
    """Device time per call (us) of the callables `calls`, captured back to back as one CUDA graph after
    three eager warm-up passes and replayed `replays` times between two events on the launching stream."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            for f in calls:
                f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for f in calls:
            f()
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (replays * len(calls))
    del g
    return us


def quantized_copies(qmm, torch, dev, gen, qt, N, K, total_bytes):
    """Copies of one N x K weight matrix (N(0, 0.02) from the seeded CUDA generator, quantized on the device)
    whose total exceeds `total_bytes`, so that consecutive calls find nothing of theirs in L2."""
    wbytes = qmm.row_bytes(qt, K) * N
    bufs = []
    for _ in range(max(2, int(total_bytes // wbytes) + 1)):
        w = torch.randn(N, K, device=dev, generator=gen) * 0.02
        b = torch.empty(wbytes, dtype=torch.uint8, device=dev)
        qmm.qmm_quantize(w, qt, N, K, b)
        bufs.append(b)
        del w
    return bufs


def case_entry(M, N, K, wbytes, xb, us, peaks):
    roof, bound = call_roofline(M, N, K, wbytes, xb, peaks)
    return {"M": M, "us": round(us, 2), "weight_gbs": round(wbytes / us / 1e3, 1),
            "tflops": round(2.0 * M * N * K / us / 1e6, 2), "frac": round(roof / us, 4), "bound": bound}


def aggregate(cases, key_w="wbytes"):
    t = sum(c["us"] for c in cases)
    r = sum(c["frac"] * c["us"] for c in cases)
    return round(r / t, 4) if t else None


PREFILL_TOKENS = [32, 64, 128, 256]


def run_moe(args, qmm, torch, dev, peaks):
    """The expert-indexed product on the MoE workload: 128 experts of 4096 x K Q4_0 (K in {512, 768, 1024}),
    top-8 routing, n tokens in {1, 2, 4, 8, 12, 16, 24}. Calls rotate through 64 id tables (8 distinct experts
    per token) and 2 expert banks (2 x 128 experts, 302-604 MB per K), so no call finds its experts in L2.
    Weights are N(0, 0.02) from torch's seeded CUDA generator (timing only), quantized on the device.
    Metric: bytes of the distinct experts each call streams / device time (CUDA events over a replayed
    graph of 64 calls); roofline per call as for the dense calls, with the distinct experts' bytes."""
    E, N, TOPK, NT, NBANK = synthetic.MOE_EXPERTS, synthetic.MOE_ROWS, synthetic.MOE_TOPK, 64, 2
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    stream = torch.cuda.Stream()
    out, prefill, tot_b, tot_t, tot_r = [], [], 0.0, 0.0, 0.0
    for K in synthetic.MOE_K:
        rb = qmm.row_bytes("Q4_0", K)
        banks = []
        for _ in range(NBANK):
            bank = []
            for _ in range(E):
                w = torch.randn(N, K, device=dev, generator=gen) * 0.02
                b = torch.empty(rb * N, dtype=torch.uint8, device=dev)
                qmm.qmm_quantize(w, "Q4_0", N, K, b)
                bank.append(b)
            banks.append(bank)
        for n in synthetic.MOE_TOKENS:
            tabs = [synthetic.expert_ids(n, batch=b) for b in range(NT)]
            idss = [torch.from_numpy(t).to(dev) for t in tabs]
            distinct = [len(np.unique(t)) for t in tabs]
            x = torch.randn(n, K, device=dev, generator=gen)
            y = torch.empty(n, TOPK, N, device=dev)
            fns = [(lambda i=i: qmm.qmm_id(banks[i % NBANK], "Q4_0", N, K, x, idss[i], y)) for i in range(NT)]
            us = time_graph(torch, stream, fns)
            wbytes = float(np.mean(distinct)) * rb * N
            t_hbm = (wbytes + n * K * 4) / (peaks["hbm_gbs"] * 1e9) * 1e6
            t_mma = 2.0 * n * TOPK * N * K / (peaks["bf16_tflops"] * 1e12) * 1e6
            roof = max(t_hbm, t_mma)
            out.append({"K": K, "n": n, "us": round(us, 2), "weight_gbs": round(wbytes / us / 1e3, 1),
                        "frac": round(roof / us, 4)})
            tot_b += wbytes
            tot_t += us
            tot_r += roof
        # prefill-sized routing, beyond the verify batches: the mat-vec expert kernel (path 1) beside the
        # tensor-core expert kernel (path 2) on the same calls
        for n in PREFILL_TOKENS:
            tabs = [synthetic.expert_ids(n, batch=b) for b in range(8)]
            idss = [torch.from_numpy(t).to(dev) for t in tabs]
            distinct = float(np.mean([len(np.unique(t)) for t in tabs]))
            x = torch.randn(n, K, device=dev, generator=gen)
            y = torch.empty(n, TOPK, N, device=dev)
            row = {"K": K, "n": n, "auto_path": qmm.qmm_id_pick_path("Q4_0", E, K, n, TOPK)}
            wbytes = distinct * rb * N
            t_roof = max((wbytes + n * K * 4) / (peaks["hbm_gbs"] * 1e9) * 1e6,
                         2.0 * n * TOPK * N * K / (peaks["bf16_tflops"] * 1e12) * 1e6)
            for path in (1, 2):
                fns = [(lambda i=i, path=path: qmm.qmm_id(banks[i % NBANK], "Q4_0", N, K, x, idss[i % 8], y,
                                                          path=path)) for i in range(16)]
                us = time_graph(torch, stream, fns)
                row["us_path%d" % path] = round(us, 2)
                row["tflops_path%d" % path] = round(2.0 * n * TOPK * N * K / us / 1e6, 2)
                row["frac_path%d" % path] = round(t_roof / us, 4)
            prefill.append(row)
        # dense routing: the same tokens routed within the first 16 experts (32-256 pairs per expert)
        for n in (64, 256, 512):
            tabs = [synthetic.expert_ids(n, E=16, topk=TOPK, batch=b) for b in range(8)]
            idss = [torch.from_numpy(t).to(dev) for t in tabs]
            x = torch.randn(n, K, device=dev, generator=gen)
            y = torch.empty(n, TOPK, N, device=dev)
            row = {"K": K, "n": n, "experts": 16, "auto_path": qmm.qmm_id_pick_path("Q4_0", E, K, n, TOPK)}
            for path in (1, 2):
                fns = [(lambda i=i, path=path: qmm.qmm_id(banks[i % NBANK], "Q4_0", N, K, x, idss[i % 8], y,
                                                          path=path)) for i in range(16)]
                us = time_graph(torch, stream, fns)
                row["us_path%d" % path] = round(us, 2)
                row["tflops_path%d" % path] = round(2.0 * n * TOPK * N * K / us / 1e6, 2)
            prefill.append(row)
        del banks
        torch.cuda.empty_cache()
    return {"metric": "expert-indexed weight-GB/s (distinct experts' bytes / time)", "unit": "GB/s",
            "value": round(tot_b / tot_t / 1e3, 1), "frac": round(tot_r / tot_t, 4),
            "workload": "2 banks x 128 experts x 4096 x K Q4_0, top-8, K in {512,768,1024}, n in "
                        "{1,2,4,8,12,16,24}; 64 id tables rotating", "cases": out,
            "prefill": {"tokens": PREFILL_TOKENS, "note": "mat-vec expert kernel (path 1) beside the tensor-core "
                        "expert kernel (path 2); auto_path is qmm_id's choice", "cases": prefill}}


def run_small_q4_0(qmm, torch, dev, peaks):
    """The small single-matrix workload: Q4_0 256 x 512, binary32 activations, 1 and 7 tokens. Its 73.7 KB of
    weights would sit in L2, so calls rotate through 2048 copies (151 MB, beyond the 129 MB L2)."""
    N, K = synthetic.SMALL_Q4_0
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    bufs = quantized_copies(qmm, torch, dev, gen, "Q4_0", N, K, 150e6)
    stream = torch.cuda.Stream()
    wbytes = qmm.row_bytes("Q4_0", K) * N
    cases = []
    for M in synthetic.SMALL_TOKENS:
        x = torch.randn(M, K, device=dev, generator=gen)
        y = torch.empty(M, N, device=dev)
        us_all = []
        for c0 in range(0, len(bufs), 256):
            fns = [(lambda b=b: qmm.qmm(b, "Q4_0", N, K, x, y)) for b in bufs[c0:c0 + 256]]
            us_all.append(time_graph(torch, stream, fns, replays=1))
        cases.append(case_entry(M, N, K, wbytes, 4, float(np.mean(us_all)), peaks))
    del bufs
    return {"workload": "Q4_0 256x512, fp32 activations, M in {1,7}; 2048 rotating weight copies (151 MB)",
            "cases": cases, "frac": aggregate(cases)}


def run_qwen3_06b(qmm, torch, dev, peaks):
    """The Qwen3-0.6B-shaped decode layer with group-64 affine 4-bit weights and bf16 activations: per token
    count M in {1, 2, 4, 8, 16}, the seven projections and the output head as one group of calls (one CUDA
    graph), weights rotating through 5 copies of the layer and head (483 MB). Metric: weight-GB/s."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    layer = synthetic.QWEN3_06B_LAYER
    ncopy = 5
    ws = {}
    for c in range(ncopy):
        for name, N, K, qt in layer:
            w = torch.randn(N, K, device=dev, generator=gen) * 0.02
            b = torch.empty(qmm.row_bytes(qt, K) * N, dtype=torch.uint8, device=dev)
            qmm.qmm_quantize(w, qt, N, K, b)
            ws[(c, name)] = b
            del w
    stream = torch.cuda.Stream()
    groups, tot_b, tot_t, tot_r = [], 0.0, 0.0, 0.0
    for M in synthetic.QWEN3_06B_TOKENS:
        xs = {K: torch.randn(M, K, device=dev, generator=gen).to(torch.bfloat16) for K in {l[2] for l in layer}}
        ys = {N: torch.empty(M, N, device=dev) for N in {l[1] for l in layer}}
        fns = [(lambda c=c, name=name, N=N, K=K, qt=qt: qmm.qmm(ws[(c, name)], qt, N, K, xs[K], ys[N]))
               for c in range(ncopy) for name, N, K, qt in layer]
        us = time_graph(torch, stream, fns) * len(layer)          # per layer pass (8 calls)
        wb = sum(qmm.row_bytes(qt, K) * N for _, N, K, qt in layer)
        roof = sum(call_roofline(M, N, K, qmm.row_bytes(qt, K) * N, 2, peaks)[0] for _, N, K, qt in layer)
        groups.append({"M": M, "us_per_layer": round(us, 2), "weight_gbs": round(wb / us / 1e3, 1),
                       "frac": round(roof / us, 4)})
        tot_b += wb
        tot_t += us
        tot_r += roof
    del ws
    return {"workload": "Qwen3-0.6B layer (q,k,v,o,gate,up,down) + lm_head 151936x1024, A4G64, bf16 "
                        "activations, M in {1,2,4,8,16}; 5 rotating copies (483 MB)",
            "value": round(tot_b / tot_t / 1e3, 1), "unit": "GB/s", "frac": round(tot_r / tot_t, 4),
            "groups": groups}


def run_sweep(qmm, torch, dev, peaks):
    """The all-type sweep on one ffn_gate-shaped 9728 x 2560 matrix, binary32 activations, M in {1, 16, 64,
    512, 2048}; per type, rotating weight copies beyond 3x L2 (400 MB); 20 calls per graph."""
    N, K = synthetic.SWEEP_SHAPE
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    stream = torch.cuda.Stream()
    out, allc = {}, []
    for qt in synthetic.SWEEP_TYPES:
        bufs = quantized_copies(qmm, torch, dev, gen, qt, N, K, 400e6)
        wbytes = qmm.row_bytes(qt, K) * N
        cases = []
        for M in synthetic.SWEEP_TOKENS:
            x = torch.randn(M, K, device=dev, generator=gen)
            y = torch.empty(M, N, device=dev)
            ws = torch.empty(max(256, qmm.qmm_workspace_size(qt, N, K, M)), dtype=torch.uint8, device=dev)
            fns = [(lambda b=bufs[i % len(bufs)]: qmm.qmm_ws(b, qt, N, K, x, y, ws)) for i in range(20)]
            cases.append(case_entry(M, N, K, wbytes, 4, time_graph(torch, stream, fns), peaks))
        out[qt] = cases
        allc += cases
        del bufs
        torch.cuda.empty_cache()
    return {"workload": "ffn_gate 9728x2560, 13 types, fp32 activations, M in {1,16,64,512,2048}",
            "frac": aggregate(allc), "types": out}


def run_unbatched(args, qmm, torch, dev, wq, peaks):
    """The layer's M <= 16 calls as seven separate qmm_ws calls (no projection batched), for comparison with
    the step's batched form. One CUDA graph per (weight copy, token count)."""
    stream = torch.cuda.Stream()
    out, tot_b, tot_t, tot_r = [], 0.0, 0.0, 0.0
    for M in (1, 2, 7):
        xs = {K: torch.from_numpy(synthetic.activations(M, K, seed=M)).to(dev) for K in {l[2] for l in LAYER}}
        ys = {name: torch.empty((M, N), dtype=torch.float32, device=dev) for name, N, K, qt in LAYER}

        def step(copy):
            for name, N, K, qt in LAYER:
                qmm.qmm_ws(wq[(copy, name)], qmm.TYPE_ID[qt] | qmm.W_STATIC, N, K, xs[K], ys[name], None)

        fns = [(lambda c=c: step(c)) for c in range(COPIES)]
        us = time_graph(torch, stream, fns, replays=max(4, args.steps // COPIES))
        wb = sum(weight_bytes(N, K, qt) for _, N, K, qt in LAYER)
        roof = sum(call_roofline(M, N, K, weight_bytes(N, K, qt), 4, peaks)[0] for _, N, K, qt in LAYER)
        out.append({"M": M, "us": round(us, 2), "weight_gbs": round(wb / us / 1e3, 1), "frac": round(roof / us, 4)})
        tot_b += wb
        tot_t += us
        tot_r += roof
    return {"metric": "weight-GB/s of the M<=16 calls, every projection its own call", "unit": "GB/s",
            "value": round(tot_b / tot_t / 1e3, 1), "frac": round(tot_r / tot_t, 4), "per_m": out}


def run_e2e(args, qmm, torch, dev, calls, wq, ws):
    """The headline metric end to end through the public API with host buffers: every step copies the
    activations of its M <= 16 calls from pinned host memory to the device (one copy of all of them), runs
    the calls through qmm_ws, and copies every call's result back to pinned host memory (one copy), all
    inside the timed region; a step is captured as one CUDA graph per weight copy, as a caller replaying a
    decode step would (weights stay resident, as a model's do)."""
    small = [c for c in calls if c[4] <= 16]
    xkeys = sorted({(c[4], c[2]) for c in small})
    xoff, nx = {}, 0
    for M, K in xkeys:
        xoff[(M, K)] = nx
        nx += M * K
    yoff, ny = [], 0
    for c in small:
        yoff.append(ny)
        ny += c[4] * c[1]
    hx = torch.empty(nx, dtype=torch.float32).pin_memory()
    for M, K in xkeys:
        hx[xoff[(M, K)]:xoff[(M, K)] + M * K] = torch.from_numpy(synthetic.activations(M, K, seed=M)).reshape(-1)
    hy = torch.empty(ny, dtype=torch.float32).pin_memory()
    dx = torch.empty(nx, dtype=torch.float32, device=dev)
    dy = torch.empty(ny, dtype=torch.float32, device=dev)

    def step(copy):
        dx.copy_(hx, non_blocking=True)
        views = {}
        for i, (name, N, K, qt, M, b) in enumerate(small):
            views[(name, M)] = (dx[xoff[(M, K)]:xoff[(M, K)] + M * K].view(M, K), dy[yoff[i]:yoff[i] + M * N].view(M, N))
        for name, N, K, qt, M, b in small:
            if name in SHARED_PARTNERS:
                continue
            x, y = views[(name, M)]
            partner = SHARED_INPUT.get(name)
            if partner:
                N2 = next(c[1] for c in small if c[0] == partner)
                qmm.qmm_batch([wq[(copy, name)], wq[(copy, partner)]], qmm.TYPE_ID[qt] | qmm.W_STATIC, [N, N2], K, x,
                              [y, views[(partner, M)][1]])
            else:
                qmm.qmm_ws(wq[(copy, name)], qmm.TYPE_ID[qt] | qmm.W_STATIC, N, K, x, y, ws)
        hy.copy_(dy, non_blocking=True)

    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for s in range(3):
            step(s % COPIES)
    torch.cuda.synchronize()
    graphs = []
    for copy in range(COPIES):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step(copy)
        graphs.append(g)
    steps = max(10, args.steps)
    with torch.cuda.stream(stream):
        for s in range(3):
            graphs[s % COPIES].replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for s in range(steps):
            graphs[s % COPIES].replay()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    wb = sum(weight_bytes(c[1], c[2], c[3]) for c in small)
    return {"value": round(wb / (ms * 1e-3) / 1e9, 1), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": nx * 4, "d2h_bytes_per_step": ny * 4, "steps": steps,
            "calls": "the 21 projections with M<=16 (q+k and gate+up batched as in the step), one host-to-device "
                     "copy of their activations and one device-to-host copy of their results per step, replayed "
                     "as CUDA graphs"}


# ---------------------------------------------------------------------------------------- oracle legs

def oracle_step_sample():
    """The bounded sample the oracle times: the seven projections at M = 1, 2 and 7 (every M <= 16 call of
    the step), on oracle-encoded copies of the same seeded weights."""
    import oracle
    ws = {}
    for name, N, K, qt in LAYER:
        ws[name] = oracle.quantize(qt, synthetic.weights(N, K, seed=0))
    xs = {(M, K): synthetic.activations(M, K, seed=M) for M in (1, 2, 7) for K in {c[2] for c in LAYER}}
    return oracle, ws, xs


def time_oracle_sample(oracle, ws, xs):
    """One pass of the oracle over the sample: every call's weights decoded to binary64 (dequant), then the
    product (matmul), the two steps timed separately. Returns (weight bytes, dequant s, matmul s)."""
    td = tm = 0.0
    wb = 0.0
    for M in (1, 2, 7):
        for name, N, K, qt in LAYER:
            t0 = time.perf_counter()
            W = oracle.dequant_f64(qt, ws[name], N, K)
            t1 = time.perf_counter()
            oracle.matmul_f64(W, xs[(M, K)])
            t2 = time.perf_counter()
            td += t1 - t0
            tm += t2 - t1
            wb += weight_bytes(N, K, qt)
    return wb, td, tm


def cpu_baseline(args, seconds=10.0):
    """The oracle on the step's 21 M<=16 calls, passes repeated for about `seconds` of CPU work."""
    oracle, ws, xs = oracle_step_sample()
    wb = td = tm = 0.0
    passes = 0
    while passes == 0 or td + tm < seconds:
        b, d, m = time_oracle_sample(oracle, ws, xs)
        wb += b
        td += d
        tm += m
        passes += 1
    t = td + tm
    return {"value": round(wb / t / 1e9, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "dequant_s": round(td, 3), "matmul_s": round(tm, 3),
            "sample": "the 21 calls with M<=16 (7 projections x M in {1,2,7}), full outputs, %d passes (%.1f s: "
                      "dequant %.1f s, matmul %.1f s)" % (passes, t, td, tm)}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    oracle, ws, xs = oracle_step_sample()
    for _ in range(args.warmup):
        time_oracle_sample(oracle, ws, xs)
    t0 = time.perf_counter()
    wb = td = tm = 0.0
    for _ in range(args.steps):
        b, d, m = time_oracle_sample(oracle, ws, xs)
        wb += b
        td += d
        tm += m
    t = time.perf_counter() - t0
    v = wb / t / 1e9
    cores = oracle.num_threads()
    sample = ("per step: the 21 calls with M<=16 of the layer (7 projections x M in {1,2,7}), full outputs; "
              "dequant %.2f s, matmul %.2f s over the run" % (td, tm))
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(world),
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
                             "dequant_s": round(td, 3), "matmul_s": round(tm, 3)},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--case", default=None, help="time one call only, e.g. ffn_gate:2048, or one expert-indexed workload, e.g. moe:256")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--detail", action="store_true", help="per-call device times on stderr")
    ap.add_argument("--no-moe", action="store_true", help="skip the expert-indexed (MoE) leg")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the small Q4_0, Qwen3-0.6B and all-type sweep objects")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
