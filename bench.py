#!/usr/bin/env python
"""Throughput of the GB300 weight-quantized linear layer.

Workload of the headline number: the decode/verify projection K = N = 5120 at
M in {1, 4, 16, 64} tokens, in both modes -- W4A16, and W4A8 with per-token
int8 activation quantization -- over 32 distinct packed weight matrices (one
per "layer", 432 MB in total, so every GEMM streams its weights from HBM, not
L2).  One step = every (mode, M) over all 32 layers: 128 W4A16 GEMMs plus 128
W4A8 layers from fp16 (one kernel up to 16 tokens; quantizer, widening and GEMM at 64).  Each (mode, M) block is captured once as a
CUDA graph through the library's public calls and replayed; CUDA events on the
launching stream time every block.

value = weight bytes streamed by the GEMMs in a step / step time (GB/s, whole
job over all ranks).  The same run reports TFLOPS/TOPS and roofline fractions
per (mode, M), and, at one GPU, the other workloads of the layer (fused FFN
pair at M=64, the M=8192 prefill, the 248k-row int8 lm_head), each with a
parity spot check against the CPU oracle.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "W4A8/W4A16 GEMM TOPS & weight-read GB/s vs M (1–8192), % of GB300 roofline"
N = K = 5120
MS = (1, 4, 16, 64)
LAYERS = 32
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "qgemm_rb_kernel_proj_w4a16_m16.md")
KERNEL_SOURCES = ("gemm_rb.cuh", "quant_code.cuh", "gemm_ms.cuh", "gemm_kernel.cuh", "ptx.cuh", "schedule.h")


def profiled_traffic():
    """DRAM bytes (read + write) of one M = 16 projection launch of the row-block decode
    kernel, from the committed ncu summary, provided the kernel sources still hash to
    what was profiled; else None."""
    try:
        text = open(TRAFFIC_PROFILE).read()
    except OSError:
        return None
    sha = re.search(r"^kernel_sources_sha256: ([0-9a-f]{64})", text, re.M)
    nbytes = re.search(r"^dram_bytes_per_launch: (\d+)", text, re.M)
    if not (sha and nbytes):
        return None
    return int(nbytes.group(1)) if sources_sha256(KERNEL_SOURCES) == sha.group(1) else None


def code_only(text: bytes) -> bytes:
    """C/C++/CUDA source without its comments and blank lines (trailing blanks dropped):
    what the compiler sees, so that a comment edit leaves a profile's link intact."""
    s = re.sub(r"/\*.*?\*/", "", text.decode(), flags=re.S)
    s = re.sub(r"//[^\n]*", "", s)
    return "\n".join(ln.rstrip() for ln in s.split("\n") if ln.strip()).encode()


def sources_sha256(files) -> str:
    """sha256 over the code (code_only) of the given csrc/ files, in that order: the
    kernel_sources_sha256 line of the summaries under profiles/."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "int8_weight_quantized_int4_gb300", "csrc", f), "rb") as fh:
            h.update(code_only(fh.read()))
    return h.hexdigest()


def w4a8_kernels(M, N, K):
    """Kernels one qgemm_w4a8_fused call launches: 1 when the quantizer runs inside
    the GEMM, else the quantizer (fp16 codes) + the GEMM."""
    import int8_weight_quantized_int4_gb300 as q
    p = q.plan(q.MODE_W4A8_FUSED, M, N, K, torch.cuda.get_device_properties(0).multi_processor_count)
    return 1 if p.fused else 2


def gemm_kernel_name(M, N, K):
    """The GEMM kernel a W4A16 call of this shape runs on (from the library's plan)."""
    import int8_weight_quantized_int4_gb300 as q
    p = q.plan(q.MODE_W4A16, M, N, K, torch.cuda.get_device_properties(0).multi_processor_count)
    return "qgemm_rb_kernel" if p.decode_row_blocks else "qgemm_ms_kernel" if p.decode_teams else "qgemm_tc_kernel"


def w4_bytes(n, k):
    return n * k // 2 + 2 * n * (k // 128)


def w8_bytes(n, k):
    return n * k + 2 * n * (k // 128)


# ------------------------------------------------------------ clocks sampler --
class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            self.path = f"/tmp/qgemm_clocks_{os.getpid()}.csv"
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.out,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- distributed --
def dist_setup(backend):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, ws, device):
    if ws == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle leg --
def oracle_sample(seconds=12.0):
    """Time the oracle, as it stands, on a bounded sample of the workload: the
    projection at each M and mode over a subset of output rows; returns
    (weight bytes covered, seconds, description)."""
    import oracle
    p = synth.projection(64)
    x = p.x
    qa, sx = oracle.quant_act_int8(x)
    # size the column sample from a short calibration run
    t0 = time.perf_counter()
    oracle.w4a16(x[:16], p.codes[:64], p.scales[:64])
    cal = (time.perf_counter() - t0) / (16 * 64 * K)
    per_col = sum(MS) * K * 2 * cal
    cols = int(max(64, min(N, seconds / max(per_col, 1e-12))))
    cols = (cols // 64) * 64
    c, s = p.codes[:cols], p.scales[:cols]
    # whole passes over the sample until the time budget is spent (at most 200)
    t0 = time.perf_counter()
    passes = 0
    while True:
        for M in MS:
            oracle.w4a16(x[:M], c, s)
            oracle.w4a8(qa[:M], sx[:M], c, s)
        passes += 1
        if time.perf_counter() - t0 >= seconds or passes >= 200:
            break
    dt = time.perf_counter() - t0
    wb = passes * 2 * len(MS) * w4_bytes(cols, K)
    desc = (f"oracle W4A16 + W4A8 at M={list(MS)} on {cols} of 5120 output rows of one "
            f"K=N=5120 layer, {passes} pass(es) ({wb / 1e6:.1f} MB of packed-weight equivalent)")
    return wb, dt, desc


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores (rank 0 only)."""
    ws, rank, _ = dist_setup("gloo")
    if rank != 0:
        return
    cores = len(os.sched_getaffinity(0))
    # per-step sample: a quarter of --cpu-seconds, shrunk so the whole run stays near
    # two and a half minutes however many steps are asked for
    budget = max(0.05, min(args.cpu_seconds / 4.0, 150.0 / (args.warmup + args.steps)))
    times, wbs, desc = [], [], ""
    for i in range(args.warmup + args.steps):
        wb, dt, desc = oracle_sample(budget)
        if i >= args.warmup:
            times.append(dt)
            wbs.append(wb)
    value = sum(wbs) / sum(times) / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * statistics.mean(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "projection K=N=5120, M in {1,4,16,64}, W4A16 + W4A8; "
                                   "bounded CPU sample per step"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm --
def time_graph(g, stream, reps=1):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for _ in range(reps):
        g.replay()
    e.record(stream)
    return s, e


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()                                    # eager warm-up: sets attributes, caches
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            fn()
    torch.cuda.synchronize()
    return g


def parity_err(y, ref):
    if isinstance(y, torch.Tensor):
        y = y.float().cpu().numpy()
    y = np.asarray(y).astype(np.float64)
    ref = np.asarray(ref).astype(np.float64)
    if not np.isfinite(y).all():
        return float("inf")
    return float(np.abs(y - ref).max() / max(np.abs(ref).max(), 1e-30))


def run_ours(args):
    import __graft_entry__
    __graft_entry__.build()
    import int8_weight_quantized_int4_gb300 as q

    ws_n, rank, local = dist_setup("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])

    # ---- inputs (seeded, synthetic), weights resident in HBM
    p = synth.projection(64)
    packed0 = q.qpack_w4(p.codes.to(dev), p.scales.to(dev))
    packed = [packed0] + [packed0.clone() for _ in range(LAYERS - 1)]
    gen = synth.generator(1000 + rank)
    X = {M: synth.activations(LAYERS * M, K, gen, outlier_frac=0.01).view(LAYERS, M, K).to(dev)
         for M in MS}
    Y16 = {M: torch.empty((LAYERS, M, N), dtype=torch.float16, device=dev) for M in MS}
    Y8 = {M: torch.empty((LAYERS, M, N), dtype=torch.float16, device=dev) for M in MS}
    wsp = q.Workspace(dev)
    for M in MS:
        for mode in (q.MODE_W4A16, q.MODE_W4A8_FUSED):
            wsp.get(mode, M, N, K)
    torch.cuda.synchronize()

    def block16(M):
        def f():
            for r in range(LAYERS):
                q.qgemm_w4a16(X[M][r], packed[r], N, K, y=Y16[M][r], ws=wsp)
        return f

    def block8(M):
        # the W4A8 layer from fp16 activations: per-token int8 quantization + GEMM
        # (one kernel for small batches, the quantizer then the GEMM otherwise)
        def f():
            for r in range(LAYERS):
                q.qgemm_w4a8_fused(X[M][r], packed[r], N, K, y=Y8[M][r], ws=wsp)
        return f

    # The same step with the library default (every kernel waits for its predecessor
    # before touching memory), reported beside the headline.
    graphs_default = [("w4a16", M, capture(block16(M), stream)) for M in MS] + \
                     [("w4a8", M, capture(block8(M), stream)) for M in MS]
    # Headline: inference on loaded weights -- the packed weights are never written by
    # the kernel before a GEMM, so each GEMM may stream them while its predecessor ends.
    torch.cuda.synchronize()
    q.set_weights_immutable(True)
    n0 = q.num_kernel_launches()
    graphs = []
    for M in MS:
        graphs.append(("w4a16", M, capture(block16(M), stream)))
    for M in MS:
        graphs.append(("w4a8", M, capture(block8(M), stream)))
    launches_per_step = (q.num_kernel_launches() - n0) // 2   # eager warm-up + capture
    step_wbytes = len(graphs) * LAYERS * w4_bytes(N, K)

    def step(events=None, gl=None):
        for mode, M, g in (graphs if gl is None else gl):
            if events is not None:
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record(stream)
                g.replay()
                e.record(stream)
                events.append((mode, M, s, e))
            else:
                g.replay()

    blocks_default = []
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step(gl=graphs_default)
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        nd = max(3, args.steps // 4)
        for _ in range(nd):
            step(blocks_default, gl=graphs_default)
        d1.record(stream)
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    value_default = step_wbytes * nd / (d0.elapsed_time(d1) / 1e3) / 1e9
    barrier(ws_n)

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.5)                                  # let the sampler start
    torch.cuda.synchronize()
    barrier(ws_n)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    blocks = []
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            step(blocks)
        t_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws_n)
    clk = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, ws_n, dev)
    ms_per_step = elapsed_ms / args.steps
    value = ws_n * step_wbytes * args.steps / (elapsed_ms / 1e3) / 1e9

    # ---- per (mode, M) figures from the block events, for the headline mode (weights
    #      declared immutable) and for the library default
    def per_m_table(blist):
        per = {}
        for mode, M, s, e in blist:
            per.setdefault((mode, M), []).append(s.elapsed_time(e))
        table = {}
        for (mode, M), v in per.items():
            ms = statistics.median(v)
            us = 1e3 * ms / LAYERS
            flops = 2.0 * M * N * K
            act_b = M * K * (2 if mode == "w4a16" else 1) + (4 * M if mode == "w4a8" else 0)
            alg = w4_bytes(N, K) + act_b + 2 * M * N
            table[f"{mode}_M{M}"] = {
                "us_per_layer": round(us, 3), "weight_GBps": round(w4_bytes(N, K) / us / 1e3, 1),
                "TFLOPS": round(flops / us / 1e6, 2), "alg_GBps": round(alg / us / 1e3, 1),
                "frac_hbm": round(alg / us / 1e3 / hbm, 4),
                "kernels_per_layer": 1 if mode == "w4a16" else w4a8_kernels(M, N, K),
                "kernel": gemm_kernel_name(M, N, K)}
        return per, table

    per, per_m = per_m_table(blocks)
    _, per_m_default = per_m_table(blocks_default)
    # roofline of the dominant kernel: the decode kernel (M <= 16, both modes), W4A16
    # launches at M = 1, 4, 16
    roof_bytes = roof_ms = 0.0
    for (mode, M), v in per.items():
        if mode == "w4a16" and M <= 16:
            roof_bytes += (w4_bytes(N, K) + 4 * M * K) * LAYERS * len(v)
            roof_ms += sum(v)
    achieved = roof_bytes / (roof_ms / 1e3) / 1e9
    traffic = profiled_traffic()
    roofline = {"bound": "hbm", "kernel": gemm_kernel_name(1, N, K) + " (W4A16, M = 1, 4, 16, K = N = 5120)",
                "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "peak_source": pk_src + " (hbm_gbs)",
                "traffic": traffic,
                "traffic_source": ("ncu capture of one M = 16 launch, DRAM read + write bytes"
                                   if traffic is not None
                                   else "null: kernel sources changed since the last ncu capture"),
                "per_launch_alg_bytes": "13,516,800 B packed weights + 2MK activation + 2MN output"}

    # ---- parity spot check of the timed outputs (the pages' lesson: a kernel can
    #      benchmark beautifully while producing garbage)
    import oracle
    parity = {}
    for M in MS:
        # every output of the last layer, and a column sample of the first
        for r, cols in ((LAYERS - 1, np.arange(N)), (0, np.arange(0, N, 7))):
            xc = X[M][r].cpu()
            ref16 = oracle.w4a16(xc, p.codes[cols], p.scales[cols])
            e16 = parity_err(Y16[M][r].cpu()[:, cols], ref16)
            oq, os_ = oracle.quant_act_int8(xc)
            ref8 = oracle.w4a8(oq, os_, p.codes[cols], p.scales[cols])
            e8 = parity_err(Y8[M][r].cpu()[:, cols], ref8)
            parity[f"w4a16_M{M}"] = max(parity.get(f"w4a16_M{M}", 0.0), e16)
            parity[f"w4a8_M{M}"] = max(parity.get(f"w4a8_M{M}", 0.0), e8)

    # ---- end to end: host (pinned) inputs in, results out, every step
    hx = {M: X[M].cpu().pin_memory() for M in MS}
    hy16 = {M: torch.empty_like(Y16[M], device="cpu").pin_memory() for M in MS}
    hy8 = {M: torch.empty_like(Y8[M], device="cpu").pin_memory() for M in MS}
    h2d = sum(hx[M].numel() * 2 for M in MS)
    d2h = sum((hy16[M].numel() + hy8[M].numel()) * 2 for M in MS)

    def e2e_step():
        for M in MS:
            X[M].copy_(hx[M], non_blocking=True)
        step()
        for M in MS:
            hy16[M].copy_(Y16[M], non_blocking=True)
            hy8[M].copy_(Y8[M], non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
        torch.cuda.synchronize()
        barrier(ws_n)
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        es.record(stream)
        for _ in range(args.steps):
            e2e_step()
        ee.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(es.elapsed_time(ee), ws_n, dev)
    e2e = {"value": round(ws_n * step_wbytes * args.steps / (e2e_ms / 1e3) / 1e9, 1), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "note": "pinned host activations in and fp16 outputs out every step, graphs of the "
                   "public calls in between"}

    derr = q.device_error()

    line = {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws_n,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic",
            "config": {"workload": "decode/verify projection K=N=5120, M in {1,4,16,64}, "
                                   "W4A16 and W4A8 (per-token int8 act quant), 32 layers",
                       "l2": "inputs larger than L2: 32 distinct 13.5 MB packed weights (432 MB) "
                             "rotate, each GEMM streams its weights from HBM",
                       "weight_bytes_per_step": step_wbytes, "graphs": True,
                       "weights_immutable_option": True,
                       "value_with_default_option": round(value_default, 1),
                       "parallelism": f"replicas x{ws_n}"},
            "roofline": roofline, "per_M": per_m, "per_M_default_option": per_m_default, "parity": parity,
            "gpu_launches": int(launches_per_step * args.steps), "clocks": clk, "e2e": e2e,
            "device_error": derr}

    print(json.dumps({k: line[k] for k in ("value", "ms_per_step", "roofline", "per_M", "parity")}),
          file=sys.stderr, flush=True)
    if ws_n == 1 and not args.no_extras:
        try:
            line["configs"] = extras(q, dev, stream, pk, pk_src)
        except Exception as ex:          # report, keep the headline line
            import traceback
            traceback.print_exc()
            line["configs"] = {"error": repr(ex)}
    if rank == 0 and ws_n == 1:
        cores = len(os.sched_getaffinity(0))
        wb, dt, desc = oracle_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(wb / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
                                "kind": "oracle", "sample": desc, "seconds": round(dt, 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def mma_rates(q, dev):
    """Dense rates of the warp-level tensor-core MMA (mma.sync) measured with the
    library's microbenchmark: every warp issues independent MMAs on register operands
    (8 chains), two 256-thread CTAs per SM, the best of 3 launches of ~20 ms each."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    res = {}
    for kind in ("f16", "s8", "e4m3", "s4"):
        iters = 2000
        best = 0.0
        for rep in range(4):
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            ops, _ = q.diag_mma_peak(kind, 2 * sms, iters, 8, dev)
            e.record()
            torch.cuda.synchronize()
            ms = s.elapsed_time(e)
            if rep == 0:
                iters = max(200, int(iters * 20.0 / max(ms, 1e-3)))
                continue
            best = max(best, ops / ms / 1e9)
        res[kind] = {"TOPS": round(best, 1), "instruction": {
            "f16": "mma.sync.m16n8k16 f16 -> f32", "s8": "mma.sync.m16n8k32 s8 -> s32",
            "e4m3": "mma.sync.m16n8k32 e4m3 -> f32", "s4": "mma.sync.m16n8k64 s4 -> s32"}[kind]}
    return res


# ----------------------------------------------------- the other workloads --
def extras(q, dev, stream, pk, pk_src):
    """FFN pair (M=64, W4A8), prefill (M=8192, both modes), 2048-token prefill chunks on
    the three layer shapes (both modes), lm_head (W8A16), the embedding gather from the
    same int8 table, top-k over logits of the lm_head's width.
    Each timed with CUDA events on graph replays, with a parity spot check."""
    import oracle
    hbm = float(pk["hbm_gbs"])
    # the prefill cells are timed over a few graph replays (milliseconds): burst peak
    peak16 = float(pk["bf16_tflops"])
    peak16_sus = float(pk.get("bf16_tflops_sustained", peak16))
    out = {}
    # measured warp-level MMA rates (the only int8 tensor-core instruction sm_103a has)
    rates = mma_rates(q, dev)
    out["mma_sync_peaks"] = rates
    int8_peak = rates["s8"]["TOPS"]

    def timeit(fn, reps):
        g = capture(fn, stream)
        with torch.cuda.stream(stream):
            for _ in range(2):
                g.replay()
            s, e = time_graph(g, stream, reps)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    # FFN pair at M=64, W4A8: up 5120 -> 34816 and down 17408 -> 5120, 4 rotating copies
    for name, prob in (("ffn_up_m64_w4a8", synth.ffn_up(64)), ("ffn_down_m64_w4a8", synth.ffn_down(64))):
        pkd = q.qpack_w4(prob.codes.to(dev), prob.scales.to(dev))
        copies = [pkd] + [pkd.clone() for _ in range(3)]
        x = prob.x.to(dev)
        y = torch.empty((64, prob.N), dtype=torch.float16, device=dev)
        wsp = q.Workspace(dev)
        wsp.get(q.MODE_W4A8_FUSED, 64, prob.N, prob.K)

        def f():
            for c in copies:
                q.qgemm_w4a8_fused(x, c, prob.N, prob.K, y=y, ws=wsp)
        ms = timeit(f, 20) / len(copies)
        wb = w4_bytes(prob.N, prob.K)
        cols = np.arange(0, prob.N, max(1, prob.N // 512))
        oq, os_ = oracle.quant_act_int8(prob.x)
        ref = oracle.w4a8(oq, os_, prob.codes[cols], prob.scales[cols])
        print(name, round(ms * 1e3, 2), "us", file=sys.stderr, flush=True)
        out[name] = {"us": round(ms * 1e3, 2), "weight_GBps": round(wb / ms / 1e6, 1),
                     "TOPS": round(2 * 64 * prob.N * prob.K / ms / 1e9, 2),
                     "frac_hbm": round((wb + 64 * prob.K + 256 + 128 * prob.N) / ms / 1e6 / hbm, 4),
                     "kernels": w4a8_kernels(64, prob.N, prob.K), "parity": parity_err(y.cpu()[:, cols], ref)}
        del copies, pkd

    # prefill M=8192, W4A16 and W4A8 on identical weights
    pp = synth.prefill(8192)
    pkd = q.qpack_w4(pp.codes.to(dev), pp.scales.to(dev))
    x = pp.x.to(dev)
    y = torch.empty((8192, pp.N), dtype=torch.float16, device=dev)
    wsp = q.Workspace(dev)
    wsp.get(q.MODE_W4A8_FUSED, 8192, pp.N, pp.K)
    flops = 2.0 * 8192 * pp.N * pp.K
    rows = np.arange(0, 8192, 61)
    cols = np.arange(0, pp.N, 211)
    for mode in ("w4a16", "w4a8"):
        if mode == "w4a16":
            f = lambda: q.qgemm_w4a16(x, pkd, pp.N, pp.K, y=y, ws=wsp)  # noqa: E731
        else:
            f = lambda: q.qgemm_w4a8_fused(x, pkd, pp.N, pp.K, y=y, ws=wsp)  # noqa: E731
        ms = timeit(f, 5)
        xr = pp.x.numpy()[rows]
        if mode == "w4a16":
            ref = oracle.w4a16(xr, pp.codes[cols], pp.scales[cols])
        else:
            oq, os_ = oracle.quant_act_int8(xr)
            ref = oracle.w4a8(oq, os_, pp.codes[cols], pp.scales[cols])
        tf = flops / ms / 1e9
        entry = {"ms": round(ms, 3), "TFLOPS": round(tf, 1), "frac_f16_peak": round(tf / peak16, 4),
                 "f16_peak_TFLOPS": peak16,
                 "peak_source": pk_src + " bf16_tflops (burst: the cell is a few ms of graph replays; "
                                         "the dense fp16 rate equals bf16)",
                 "frac_f16_sustained_peak": round(tf / peak16_sus, 4),
                 "parity": parity_err(y.cpu().numpy()[rows][:, cols], ref)}
        if mode == "w4a8":
            # the int8 x int4 products run exactly on the fp16 tensor path; against the
            # measured int8 tensor rate (mma.sync s8) the fraction exceeds 1
            entry.update({"TOPS": round(tf, 1), "int8_peak": round(int8_peak, 1),
                          "int8_peak_source": "mma.sync m16n8k32 s8 microbenchmark in this run",
                          "frac_int8_peak": round(tf / int8_peak, 3)})
        out[f"prefill_m8192_{mode}"] = entry
    del pkd, x, y, wsp
    torch.cuda.empty_cache()

    # 2048-token prefill chunks (the serving stack's chunk size) on the three layer shapes
    for name, prob in (("proj", synth.projection(2048)), ("ffn_up", synth.ffn_up(2048)),
                       ("ffn_down", synth.ffn_down(2048))):
        pkd = q.qpack_w4(prob.codes.to(dev), prob.scales.to(dev))
        x = prob.x.to(dev)
        y = torch.empty((2048, prob.N), dtype=torch.float16, device=dev)
        wsp = q.Workspace(dev)
        for mode in (q.MODE_W4A16, q.MODE_W4A8_FUSED):
            wsp.get(mode, 2048, prob.N, prob.K)
        flops = 2.0 * 2048 * prob.N * prob.K
        rows = np.arange(0, 2048, 97)
        cols = np.arange(0, prob.N, max(1, prob.N // 256))
        xr = prob.x.numpy()[rows]
        for mode in ("w4a16", "w4a8"):
            if mode == "w4a16":
                f = lambda: q.qgemm_w4a16(x, pkd, prob.N, prob.K, y=y, ws=wsp)  # noqa: E731
                ref = oracle.w4a16(xr, prob.codes[cols], prob.scales[cols])
            else:
                f = lambda: q.qgemm_w4a8_fused(x, pkd, prob.N, prob.K, y=y, ws=wsp)  # noqa: E731
                oq, os_ = oracle.quant_act_int8(xr)
                ref = oracle.w4a8(oq, os_, prob.codes[cols], prob.scales[cols])
            ms = timeit(f, 10)
            tf = flops / ms / 1e9
            out[f"prefill_chunk_m2048_{name}_{mode}"] = {
                "us": round(ms * 1e3, 1), "TFLOPS": round(tf, 1), "frac_f16_peak": round(tf / peak16, 4),
                "peak": "bf16_tflops burst",
                "N": prob.N, "K": prob.K, "parity": parity_err(y.cpu().numpy()[rows][:, cols], ref)}
        del pkd, x, y, wsp
    torch.cuda.empty_cache()

    def lm_head_topk(mode, x, pk, N, K, gemm_ms, ws):
        # the lm_head with its top-k fused in, against the plain GEMM alone and against the
        # GEMM followed by the standalone top-k; exactness of the fused top-k vs the oracle
        k, M = 64, x.shape[0]
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        v = torch.empty((M, k), dtype=torch.float16, device=dev)
        i = torch.empty((M, k), dtype=torch.int32, device=dev)
        wst = q.Workspace(dev)
        fused = lambda: q.qgemm_lm_head_topk(mode, x, pk, N, K, k, y=y, vals=v, idx=i, ws=wst)  # noqa: E731
        ms_f = timeit(fused, 10)
        gemm = q.qgemm_w4a16 if mode == q.MODE_W4A16 else q.qgemm_w8a16

        def separate():
            gemm(x, pk, N, K, y=y, ws=ws)
            q.topk_logits(y, k)
        ms_s = timeit(separate, 10)
        fused()
        torch.cuda.synchronize()
        ov, oi = oracle.topk(y.cpu().numpy(), k)
        exact = bool(np.array_equal(i.cpu().numpy().astype(np.int64), oi) and
                     np.array_equal(v.cpu().numpy().view(np.uint16), ov.view(np.uint16)))
        return {"us": round(ms_f * 1e3, 1), "gemm_us": round(gemm_ms * 1e3, 1),
                "added_us": round((ms_f - gemm_ms) * 1e3, 2), "separate_us": round(ms_s * 1e3, 1),
                "k": k, "exact": exact}

    # lm_head W8A16: 248,320 x 5120 int8 (1.29 GB > L2)
    lh = synth.lm_head(64)
    pk8 = q.qpack_w8(lh.codes.to(dev), lh.scales.to(dev))
    wb = w8_bytes(lh.N, lh.K)
    cols = np.concatenate([np.arange(0, lh.N, 997), [lh.N - 1]])
    wsp = q.Workspace(dev)
    for M in (1, 8, 16, 64):
        x = lh.x[:M].contiguous().to(dev)
        y = torch.empty((M, lh.N), dtype=torch.float16, device=dev)
        wsp.get(q.MODE_W8A16, M, lh.N, lh.K)
        ms = timeit(lambda: q.qgemm_w8a16(x, pk8, lh.N, lh.K, y=y, ws=wsp), 10)
        ref = oracle.w8a16(lh.x[:M], lh.codes[cols], lh.scales[cols])
        alg = wb + 2 * M * lh.K + 2 * M * lh.N
        out[f"lm_head_w8a16_M{M}"] = {"us": round(ms * 1e3, 1), "weight_GBps": round(wb / ms / 1e6, 1),
                                      "frac_hbm": round(alg / ms / 1e6 / hbm, 4),
                                      "TFLOPS": round(2 * M * lh.N * lh.K / ms / 1e9, 2),
                                      "parity": parity_err(y.cpu()[:, cols], ref)}
        if M in (1, 16, 64):
            out[f"lm_head_topk_w8a16_M{M}"] = lm_head_topk(q.MODE_W8A16, x, pk8, lh.N, lh.K, ms, wsp)

    # dequant-on-gather from the same int8 group-128 table (the embedding's format)
    for T in (64, 2048):
        ids = synth.token_ids(T, lh.N, seed=40 + T).to(dev)
        emb = torch.empty((T, lh.K), dtype=torch.float16, device=dev)
        ms = timeit(lambda: q.embed_gather_w8(ids, pk8, lh.N, lh.K, out=emb), 20)
        sel = np.arange(0, T, max(1, T // 16))
        ref = oracle.embed_w8(ids.cpu().numpy()[sel], lh.codes, lh.scales)
        moved = T * (lh.K + 2 * lh.K // 128) + 2 * T * lh.K
        out[f"embed_gather_w8_T{T}"] = {
            "us": round(ms * 1e3, 2), "GBps": round(moved / ms / 1e6, 1),
            "bitexact_sampled_rows": bool(np.array_equal(emb.cpu().numpy()[sel].view(np.uint16),
                                                         ref.view(np.uint16)))}
    del pk8
    torch.cuda.empty_cache()

    # int4 lm_head (W4A16 at the vocabulary width): 248,320 x 5120 int4, 655 MB packed
    l4 = synth.lm_head_int4(64)
    pk4 = q.qpack_w4(l4.codes.to(dev), l4.scales.to(dev))
    wb4 = w4_bytes(l4.N, l4.K)
    cols4 = np.concatenate([np.arange(0, l4.N, 997), [l4.N - 1]])
    for M in (1, 16, 64):
        x = l4.x[:M].contiguous().to(dev)
        y = torch.empty((M, l4.N), dtype=torch.float16, device=dev)
        wsp.get(q.MODE_W4A16, M, l4.N, l4.K)
        ms = timeit(lambda: q.qgemm_w4a16(x, pk4, l4.N, l4.K, y=y, ws=wsp), 10)
        ref = oracle.w4a16(l4.x[:M], l4.codes[cols4], l4.scales[cols4])
        alg = wb4 + 2 * M * l4.K + 2 * M * l4.N
        out[f"lm_head_w4a16_M{M}"] = {"us": round(ms * 1e3, 1), "weight_GBps": round(wb4 / ms / 1e6, 1),
                                      "frac_hbm": round(alg / ms / 1e6 / hbm, 4),
                                      "TFLOPS": round(2 * M * l4.N * l4.K / ms / 1e9, 2),
                                      "parity": parity_err(y.cpu()[:, cols4], ref)}
        out[f"lm_head_topk_w4a16_M{M}"] = lm_head_topk(q.MODE_W4A16, x, pk4, l4.N, l4.K, ms, wsp)
    del pk4, l4
    torch.cuda.empty_cache()

    # int8-QK causal prefill attention, head_dim 256, 24 query heads on 4 KV heads: a full
    # 4k prefill and a 2k chunk at the end of a 16k context; parity on the last 128
    # queries of one query head per KV head
    import oracle.attention as attn_oracle
    for T, S in ((4096, 4096), (2048, 16384)):
        Hq, Hkv = 24, 4
        qq, kk, vv = synth.attention(T, S, Hq, Hkv, seed=60 + T)
        qd, kd, vd = qq.to(dev), kk.to(dev), vv.to(dev)
        o = torch.empty((T, Hq, 256), dtype=torch.float16, device=dev)
        wsa = q.Workspace(dev)
        ms = timeit(lambda: q.attn_int8qk_prefill(qd, kd, vd, out=o, ws=wsa), 10)
        pos = np.arange(T, dtype=np.float64) + (S - T)
        flops = 4.0 * 256 * Hq * float((pos + 1).sum())      # QK^T and P.V over the causal triangle
        heads = [h * (Hq // Hkv) for h in range(Hkv)]
        ref = attn_oracle.attn_int8qk(qq[-128:, heads].numpy(), kk.numpy(), vv.numpy(), out_f64=True)
        got = o[-128:, heads].float().cpu().numpy()
        tf = flops / ms / 1e9
        out[f"attn_int8qk_T{T}_S{S}_Hq{Hq}_Hkv{Hkv}"] = {
            "us": round(ms * 1e3, 1), "TFLOPS": round(tf, 1), "frac_f16_peak": round(tf / peak16, 4),
            "peak": "bf16_tflops burst", "parity": float(np.abs(got - ref).max() / np.abs(ref).max())}
        del qd, kd, vd, o, wsa
    torch.cuda.empty_cache()

    # top-k (k = 64) over synthetic logits of the lm_head's width
    for M in (1, 16, 64):
        lg = synth.logits(M, lh.N, seed=50 + M).to(dev)
        ms = timeit(lambda: q.topk_logits(lg, 64), 20)
        entry = {"us": round(ms * 1e3, 2), "GBps": round(2 * M * lh.N / ms / 1e6, 1), "k": 64}
        v, i = q.topk_logits(lg, 64)
        ov, oi = oracle.topk(lg.cpu().numpy(), 64)
        entry["exact"] = bool(np.array_equal(i.cpu().numpy().astype(np.int64), oi) and
                              np.array_equal(v.cpu().numpy().view(np.uint16), ov.view(np.uint16)))
        out[f"topk_logits_M{M}_N{lh.N}"] = entry
    return out


NCU_CASES = {
    # name: (mode, M, N, K, bits)
    "proj_w4a16_m1": ("w4a16", 1, 5120, 5120, 4),
    "proj_w4a16_m16": ("w4a16", 16, 5120, 5120, 4),
    "proj_w4a16_m64": ("w4a16", 64, 5120, 5120, 4),
    "proj_w4a8_m16": ("w4a8", 16, 5120, 5120, 4),
    "proj_w4a8_fused_m4": ("w4a8f", 4, 5120, 5120, 4),
    "ffn_up_w4a8_m64": ("w4a8", 64, 34816, 5120, 4),
    "lm_head_w8a16_m16": ("w8a16", 16, 248320, 5120, 8),
    "lm_head_w4a16_m1": ("w4a16", 1, 248320, 5120, 4),
    "lm_head_w4a16_m16": ("w4a16", 16, 248320, 5120, 4),
    "ffn_up_w4a16_m64": ("w4a16", 64, 34816, 5120, 4),
    "prefill_w4a16_m2048": ("w4a16", 2048, 34816, 5120, 4),
    "prefill_w4a8_m2048": ("w4a8", 2048, 34816, 5120, 4),
    # top-k (k = 64) over M rows of N logits: ("topk", M, N, k, 0)
    "topk_m64": ("topk", 64, 248320, 64, 0),
    # dequant-on-gather of T rows from the int8 group-128 table: ("gather", T, V, D, 8)
    "embed_gather_t2048": ("gather", 2048, 248320, 5120, 8),
    # int8-QK prefill attention: ("attn", T, S, Hq, Hkv)
    "attn_t1024_s4096": ("attn", 1024, 4096, 24, 4),
    # the lm_head with the fused top-k (k = 64): ("lmtopk", M, N, K, bits)
    "lm_head_topk_w4a16_m16": ("lmtopk", 16, 248320, 5120, 4),
}


def run_ncu_case(name):
    """A small case for profiler captures: 3 eager warm-up launches of one kernel,
    then the launch to capture (the 4th launch of that kernel in the process)."""
    import __graft_entry__
    __graft_entry__.build()
    import int8_weight_quantized_int4_gb300 as q
    mode, M, N, K, bits = NCU_CASES[name]
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    if mode == "gather":
        p = synth.make_problem(1, N, K, seed=5, bits=8, scale_lo=0.001, scale_hi=0.01)
        packed = q.qpack_w8(p.codes.to(dev), p.scales.to(dev))
        ids = synth.token_ids(M, N, seed=40 + M).to(dev)
        for _ in range(4):
            out = q.embed_gather_w8(ids, packed, N, K)
        torch.cuda.synchronize()
        assert q.device_error() == 0
        print(json.dumps({"ncu_case": name, "T": M, "V": N, "D": K, "absmax": float(out.float().abs().max())}))
        return
    if mode == "attn":
        T, S, Hq, Hkv = M, N, K, bits
        qq, kk, vv = synth.attention(T, S, Hq, Hkv, seed=60 + T)
        qd, kd, vd = qq.to(dev), kk.to(dev), vv.to(dev)
        for _ in range(4):
            o = q.attn_int8qk_prefill(qd, kd, vd)
        torch.cuda.synchronize()
        assert q.device_error() == 0
        print(json.dumps({"ncu_case": name, "T": T, "S": S, "absmax": float(o.float().abs().max())}))
        return
    if mode == "lmtopk":
        p = synth.lm_head_int4(M)
        packed = q.qpack_w4(p.codes.to(dev), p.scales.to(dev))
        x = p.x.to(dev)
        for _ in range(4):
            y, vals, idx = q.qgemm_lm_head_topk(q.MODE_W4A16, x, packed, N, K, 64)
        torch.cuda.synchronize()
        assert q.device_error() == 0
        print(json.dumps({"ncu_case": name, "M": M, "idx0": int(idx[0, 0])}))
        return
    if mode == "topk":
        lg = synth.logits(M, N, seed=50 + M).to(dev)
        for _ in range(4):
            vals, idx = q.topk_logits(lg, K)
        torch.cuda.synchronize()
        assert q.device_error() == 0
        print(json.dumps({"ncu_case": name, "M": M, "N": N, "k": K, "idx0": int(idx[0, 0])}))
        return
    p = synth.make_problem(M, N, K, seed=1, bits=bits, outlier_frac=0.01)
    packed = (q.qpack_w4 if bits == 4 else q.qpack_w8)(p.codes.to(dev), p.scales.to(dev))
    x = p.x.to(dev)
    ws = q.Workspace(dev)
    if mode == "w4a8":
        xq, xs = q.quant_act_int8(x)
        fn = lambda: q.qgemm_w4a8(xq, xs, packed, N, K, ws=ws)  # noqa: E731
    elif mode == "w4a8f":
        fn = lambda: q.qgemm_w4a8_fused(x, packed, N, K, ws=ws)  # noqa: E731
    elif mode == "w8a16":
        fn = lambda: q.qgemm_w8a16(x, packed, N, K, ws=ws)  # noqa: E731
    else:
        fn = lambda: q.qgemm_w4a16(x, packed, N, K, ws=ws)  # noqa: E731
    for _ in range(4):
        y = fn()
    torch.cuda.synchronize()
    assert q.device_error() == 0
    print(json.dumps({"ncu_case": name, "M": M, "N": N, "K": K, "mode": mode,
                      "y_absmax": float(y.float().abs().max())}))


def e4m3_of_int(v):
    """The e4m3 byte of each integer (|v| <= 448 with at most 4 significant bits, which
    every int4 code and every 16 h, l half of an int8 code satisfies), from the format:
    sign, 4-bit exponent biased by 7, 3-bit mantissa."""
    v = np.asarray(v, dtype=np.int64)
    sign = (v < 0).astype(np.uint8) << 7
    a = np.abs(v)
    out = np.zeros(a.shape, np.uint8)
    nz = a > 0
    e = np.floor(np.log2(np.maximum(a, 1))).astype(np.int64)
    m = a * 8 // (1 << e) - 8
    if not np.all((a[nz] * 8) % (1 << e[nz]) == 0):
        raise ValueError("value needs more than 4 significant bits")
    out[nz] = (((e[nz] + 7) << 3) | m[nz]).astype(np.uint8)
    return out | sign


def run_diag(args):
    """Measurement tools behind the design choices: warp-level MMA rates (8 chains) and
    latencies (1 chain), tcgen05.mma issue time and completion latency at the GEMM's
    shapes, and whether int4 x int8 products split into e4m3 terms come out exact on
    tcgen05 kind::f8f6f4.  One JSON line."""
    import __graft_entry__
    __graft_entry__.build()
    import int8_weight_quantized_int4_gb300 as q
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"sms": sms, "mma_sync": {}, "tcgen05": {}, "f8f6f4_exact": {}}
    clocks = Clocks(0)
    clocks.start()
    for kind in ("f16", "s8", "e4m3", "s4"):
        for chains in (8, 1):
            iters, best, per_iter = 2000, 0.0, 0.0
            for rep in range(4):
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record()
                ops, _ = q.diag_mma_peak(kind, 2 * sms if chains == 8 else sms, iters, chains, dev)
                e.record()
                torch.cuda.synchronize()
                ms = s.elapsed_time(e)
                if rep == 0:
                    iters = max(200, int(iters * 20.0 / max(ms, 1e-3)))
                    continue
                if ops / ms / 1e9 > best:
                    best, per_iter = ops / ms / 1e9, ms * 1e6 / iters
            out["mma_sync"][f"{kind}_chains{chains}"] = {"TOPS": round(best, 1), "ns_per_iteration": round(per_iter, 2)}
    # kind + 2: the warp-collective issue form (the library's kernels); without it lane 0
    # issues alone inside a divergent branch
    for name, kind, a_tmem, n, issuers, chunks, window in (
            ("f16_A_tmem_n16_1issuer_wait_each", 0, 1, 16, 1, 64, 1),
            ("f16_A_tmem_n16_4issuers_no_wait", 0, 1, 16, 4, 256, 0),
            ("f16_A_smem_n16_1issuer_wait_each", 0, 0, 16, 1, 64, 1),
            ("f8f6f4_A_tmem_n16_1issuer_wait_each", 1, 1, 16, 1, 64, 1),
            ("f16_A_tmem_n256_dense", 0, 1, 256, 1, 2048, 0),
            ("f8f6f4_A_tmem_n256_dense", 1, 1, 256, 1, 2048, 0),
            ("warp_f16_A_tmem_n16_1issuer_wait_each", 2, 1, 16, 1, 64, 1),
            ("warp_f16_A_tmem_n16_1issuer_window4", 2, 1, 16, 1, 2048, 4),
            ("warp_f16_A_tmem_n64_1issuer_window4", 2, 1, 64, 1, 2048, 4),
            ("warp_f16_A_smem_n64_1issuer_window4", 2, 0, 64, 1, 2048, 4),
            ("warp_f16_A_tmem_n128_1issuer_window4", 2, 1, 128, 1, 2048, 4),
            ("warp_f16_A_tmem_n256_dense", 2, 1, 256, 1, 2048, 0),
            ("warp_f8f6f4_A_tmem_n256_dense", 3, 1, 256, 1, 2048, 0),
            ("f16_A_tmem_n64_1issuer_window4", 0, 1, 64, 1, 2048, 4)):
        q.diag_tc_probe(kind, a_tmem, n, issuers, chunks, window, sms)
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        o = q.diag_tc_probe(kind, a_tmem, n, issuers, chunks, window, sms)
        e.record()
        torch.cuda.synchronize()
        ms = s.elapsed_time(e)
        a = o.cpu().numpy().astype(np.float64)[:, :issuers, :]
        done = a[..., 3].sum()
        nmma = 8 if kind % 2 == 0 else 4
        out["tcgen05"][name] = {
            "issue_ns_per_mma": round(float(a[..., 0].sum() / done / nmma), 1),
            "wait_ns_per_chunk": round(float(a[..., 1].sum() / done), 1),
            "ns_per_chunk_per_cta": round(float(a[..., 2].max(axis=1).mean() / (chunks * issuers)), 1),
            "TFLOPS": round(2.0 * 128 * n * 128 * chunks * issuers * sms / ms / 1e9, 1)}
    rng = np.random.default_rng(0)
    for K in (256, 512):
        qw = rng.integers(-8, 8, (128, K // 2))
        qa = rng.integers(-127, 128, (16, K // 2))
        A = np.repeat(qw, 2, axis=1)
        B = np.stack([16 * (qa >> 4), qa & 15], axis=2).reshape(16, K)
        ref = qw.astype(np.int64) @ qa.T.astype(np.int64)
        for a_tmem in (0, 1):
            d = q.diag_f8f6f4_gemm(torch.from_numpy(e4m3_of_int(A)).to(dev), torch.from_numpy(e4m3_of_int(B)).to(dev),
                                   bool(a_tmem))
            torch.cuda.synchronize()
            out["f8f6f4_exact"][f"K{K}_A_{'tmem' if a_tmem else 'smem'}"] = bool(
                np.array_equal(d.cpu().numpy().astype(np.float64), ref.astype(np.float64)))
    out["clocks"] = clocks.stop()
    out["device_error"] = q.device_error()
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--ncu-case", choices=sorted(NCU_CASES), default=None,
                    help="run one small GEMM case for a profiler capture and exit")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--diag", action="store_true", help="run the MMA microbenchmarks and probes and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.diag:
        run_diag(args)
    elif args.ncu_case:
        run_ncu_case(args.ncu_case)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
