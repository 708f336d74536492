"""Benchmark of the quantized scaled-GEMM hot path on GB300.

Default workload (one "step"): the block-FP8 W8A8 linear with weight blocks
[128, 128], W e4m3 [18432, 7168], for a batch of activations at every token
count M in {1, 8, 17, 128, 1024, 4096}: per M, per-token-group quantization
of the bf16 activations followed by the scaled GEMM.  The metric is the
whole-job throughput in TFLOP/s (2*M*N*K summed over the six GEMMs, divided
by the step time).  Inputs are seeded synthetic data; every GEMM of a step
reads its own copy of W (6 distinct 132 MB copies), so no GEMM finds its
weights in the 129 MB L2.

Other workloads (--workload) measure the remaining hot-path configurations
for the results tables; the default line is the contract line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

N_W, K_W = 18432, 7168
# DRAM bytes (read + write) of one launch of the dominant kernel, from
# `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none
#  -k regex:gemm_kernel -s 1 -c 1 python bench.py --profile 4096`
# (summarised in profiles/); set to None whenever that kernel changes.
DOMINANT_KERNEL = "gemm_kernel<F8F8, NORMAL, 128, promote> (M=4096)"
DOMINANT_TRAFFIC_BYTES = 164.238848e6 + 125.967360e6
M_SET = (1, 8, 17, 128, 1024, 4096)
METRIC = "FP8 block-scaled W8A8 linear (quant + scaled GEMM) throughput, [128,128] weights"
WORKLOAD = ("block-FP8 W8A8 linear, W e4m3 [18432, 7168] with [128,128] fp32 block scales, "
            "bf16 activations M in {1,8,17,128,1024,4096} quantized per 1x128 group")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class Clocks:
    """Samples nvidia-smi during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            p = [x.strip() for x in l.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
            except ValueError:
                continue
            for name, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- workloads

def make_block128_inputs(dev, seed_base=0):
    from mxfp4_quantized_gemm_token_gb300 import synth
    ws_list = [synth.block_fp8_weight(N_W, K_W, 128, seed=seed_base + i, device=dev)
               for i in range(len(M_SET))]
    xs = [synth.activations(M, K_W, seed=1000 + M, device=dev) for M in M_SET]
    return ws_list, xs


def step_block128(mxq, ws_list, xs, outs, workspaces, dom_events=None):
    for i, M in enumerate(M_SET):
        wq, wsc = ws_list[i]
        q, s = mxq.per_token_group_quant_fp8(xs[i])
        if dom_events is not None and M == M_SET[-1]:
            dom_events[0].record()
        outs[i] = mxq.fp8_scaled_mm(q, wq, wsc, [128, 128], a_scale=s, workspace=workspaces[i])
        if dom_events is not None and M == M_SET[-1]:
            dom_events[1].record()


def flops_block128():
    return sum(2.0 * M * N_W * K_W for M in M_SET)


_ORACLE_INPUTS = []


def cpu_oracle_sample(seconds: float = 12.0, max_rows: int = 512):
    """The oracle (plain C, fp64) on a bounded sample of the default workload:
    whole rows of the M = 4096 GEMM (activation quantization + all 18432
    outputs of each row), rows added until the time budget is spent."""
    import oracle
    oracle.build()
    if not _ORACLE_INPUTS:
        from mxfp4_quantized_gemm_token_gb300 import synth
        wq, ws = synth.block_fp8_weight(N_W, K_W, 128, seed=0)
        x = synth.activations(512, K_W, seed=1000 + 4096)
        _ORACLE_INPUTS.extend([wq.view(torch.uint8).numpy(), ws.numpy(),
                               x.view(torch.int16).numpy().view(np.uint16)])
    w_np, ws_np, xb = _ORACLE_INPUTS
    rows, t_total = 0, 0.0
    while rows < max_rows and t_total < seconds:
        t0 = time.perf_counter()
        q, s = oracle.per_token_group_quant_fp8(xb[rows:rows + 1], 128)
        oracle.scaled_mm(q, oracle.E4M3, s, w_np, ws_np, 128, 128)
        t_total += time.perf_counter() - t0
        rows += 1
    flops = 2.0 * rows * N_W * K_W
    return {"value": flops / t_total / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": "%d full rows (quant + 18432 outputs each) of the M=4096 GEMM, %.1f s"
                      % (rows, t_total)}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    steps = []
    for _ in range(args.warmup):
        cpu_oracle_sample(seconds=2.0, max_rows=2)
    t0 = time.perf_counter()
    res = None
    for _ in range(args.steps):
        res = cpu_oracle_sample(seconds=max(3.0, 20.0 / max(1, args.steps)), max_rows=512)
        steps.append(res["value"])
    elapsed = time.perf_counter() - t0
    v = statistics.mean(steps)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * elapsed / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": res["sample"] if res else None},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": res["cores"] if res else None,
                             "kind": "oracle", "sample": res["sample"] if res else None},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args, world, rank, local):
    import mxfp4_quantized_gemm_token_gb300 as mxq
    dev = torch.device("cuda", local)
    pk, pk_src = peaks()
    ws_list, xs = make_block128_inputs(dev)
    outs = [None] * len(M_SET)
    workspaces = []
    launches_per_step = 0
    import ctypes
    lib = mxq._lib.load()
    for M in M_SET:
        sz = ctypes.c_size_t(0)
        mxq.check(lib.mxq_fp8_scaled_mm_workspace_size(M, N_W, K_W, 3, 128, 128,
                                                            ctypes.byref(sz)))
        workspaces.append(torch.empty(sz.value, dtype=torch.uint8, device=dev) if sz.value else None)
        launches_per_step += 2 + (1 if sz.value else 0)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        step_block128(mxq, ws_list, xs, outs, workspaces)
    mxq.sync_status(dev)
    torch.cuda.synchronize()

    dom = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        start.record()
        for k in range(args.steps):
            step_block128(mxq, ws_list, xs, outs, workspaces, dom_events=dom[k])
        end.record()
        torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(world, start.elapsed_time(end))
    mxq.sync_status(dev)
    ms_step = ms_total / args.steps
    flops = flops_block128()
    value = world * flops / (ms_step * 1e-3) / 1e12
    dom_ms = statistics.mean(a.elapsed_time(b) for a, b in dom)
    dom_flops = 2.0 * M_SET[-1] * N_W * K_W
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    fp8_peak = 2.0 * pk["bf16_tflops"]          # e4m3 = 2 x bf16 (nominal ratio 4.5 / 2.25)

    # ---- end to end: host activations in, host outputs back, through the API
    pinned_in = [x.cpu().pin_memory() for x in xs]
    pinned_out = [torch.empty((M, N_W), dtype=torch.bfloat16).pin_memory() for M in M_SET]
    h2d = sum(t.numel() * t.element_size() for t in pinned_in)
    d2h = sum(t.numel() * t.element_size() for t in pinned_out)
    dev_in = [torch.empty_like(x) for x in xs]
    # Three streams, pipelined across the six GEMMs of a step (and across
    # steps): host->device copies of the next inputs and device->host copies
    # of earlier results overlap the quant + GEMM of the current one.  Every
    # step still moves all of its inputs in and all of its results out.
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in M_SET]     # input i is on the device
    ev_q = [torch.cuda.Event() for _ in M_SET]      # input i consumed (quantized)
    ev_c = [torch.cuda.Event() for _ in M_SET]      # result i computed

    def e2e_step():
        for i, M in enumerate(M_SET):
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_q[i])            # the previous step read dev_in[i]
                dev_in[i].copy_(pinned_in[i], non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[i])
                q, s = mxq.per_token_group_quant_fp8(dev_in[i])
                ev_q[i].record(s_cmp)
                o = mxq.fp8_scaled_mm(q, ws_list[i][0], ws_list[i][1], [128, 128], a_scale=s,
                                      workspace=workspaces[i])
                ev_c[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c[i])
                pinned_out[i].copy_(o, non_blocking=True)
                o.record_stream(s_out)

    main = torch.cuda.current_stream(dev)

    def fork():
        for st in (s_in, s_cmp, s_out):
            st.wait_stream(main)

    def join():
        for st in (s_in, s_cmp, s_out):
            main.wait_stream(st)

    fork()
    for _ in range(max(1, args.warmup)):
        e2e_step()
    join()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    fork()
    for _ in range(args.steps):
        e2e_step()
    join()
    e1.record(main)
    torch.cuda.synchronize()
    # the pipelined copies returned exactly what the device-resident steps computed
    for i in range(len(M_SET)):
        if not torch.equal(pinned_out[i], outs[i].cpu()):
            raise RuntimeError("end-to-end result for M=%d differs from the device run" % M_SET[i])
    barrier(world)
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1)) / args.steps
    e2e_value = world * flops / (e2e_ms * 1e-3) / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3 x fp8_e4m3 -> f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": list(M_SET), "N": N_W, "K": K_W,
                   "weight_block": [128, 128], "activation_group": 128,
                   "l2": "6 distinct 132 MB weight copies, one per GEMM of a step",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": achieved / fp8_peak,
                     "traffic": DOMINANT_TRAFFIC_BYTES,
                     "kernel": DOMINANT_KERNEL,
                     "peak_source": "%s bf16 burst %.1f TFLOP/s x 2 (e4m3/bf16 nominal)"
                                    % (pk_src, pk["bf16_tflops"]),
                     "launch_ms": dom_ms},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "overlap": "h2d / compute / d2h on three streams, pipelined over the six GEMMs"},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if args.traffic is not None:
        line["roofline"]["traffic"] = args.traffic
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_profile(args, local):
    """A few launches of one shape (for ncu captures): quant + GEMM at M."""
    import mxfp4_quantized_gemm_token_gb300 as mxq
    from mxfp4_quantized_gemm_token_gb300 import synth
    dev = torch.device("cuda", local)
    M = args.profile
    wq, wsc = synth.block_fp8_weight(N_W, K_W, 128, seed=0, device=dev)
    x = synth.activations(M, K_W, seed=1000 + M, device=dev)
    for _ in range(3):
        q, s = mxq.per_token_group_quant_fp8(x)
        out = mxq.fp8_scaled_mm(q, wq, wsc, [128, 128], a_scale=s)
    torch.cuda.synchronize()
    mxq.sync_status(dev)
    print(json.dumps({"profile_M": M, "checksum": float(out.float().abs().sum().item())}))
    return 0


# ---------------------------------------------------------- other workloads

class L2Flush:
    """Evicts L2 before a timed call by reading a 512 MB buffer (4x L2).  A
    read leaves only clean lines behind; a write flush would leave ~L2-size
    dirty lines whose write-back then overlaps the timed call."""

    def __init__(self, dev, mode="read"):
        self.buf = torch.zeros(128 * 1024 * 1024, dtype=torch.float32, device=dev)
        self.acc = torch.zeros((), dtype=torch.float32, device=dev)
        self.mode = mode

    def __call__(self):
        if self.mode == "write":
            self.buf.zero_()
        else:
            torch.sum(self.buf, dim=0, out=self.acc)


def _timed_calls(fn, reps, flush):
    """Median device time (ms) of fn() over reps calls, L2 flushed before each."""
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def run_profile_moe(args, local):
    """Two fused-MoE calls of one shape, for ncu captures of the MoE kernels:
    --profile-moe fp8:T:E (FP8-block, topk 8, K 7168, N 2048) or
    mxfp4:T:E (MXFP4 + bias, topk 4, K = N = 2880); uniform routing."""
    import mxfp4_quantized_gemm_token_gb300 as mxq
    from mxfp4_quantized_gemm_token_gb300 import synth
    dev = torch.device("cuda", local)
    kind, T, E = args.profile_moe.split(":")
    T, E = int(T), int(E)
    if kind == "fp8":
        topk, K, N = 8, 7168, 2048
        w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=0, device=dev)
        kw = {}
    else:
        topk, K, N = 4, 2880, 2880
        w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=0, device=dev)
        b1, b2 = synth.moe_biases(E, N, K, seed=1, device=dev)
        kw = dict(wtype=mxq.W_MXFP4, w1_bias=b1, w2_bias=b2)
    tw, ids = synth.routing_uniform(T, E, topk, seed=T)
    x = synth.activations(T, K, seed=T, scale_div=10, device=dev)
    tw, ids = tw.to(dev), ids.to(dev)
    for _ in range(2):
        mxq.fused_experts(x, w1, s1, w2, s2, tw, ids, block_m=args.block_m, **kw)
    mxq.sync_status(dev)
    print(json.dumps({"profile_moe": args.profile_moe, "experts_touched": synth.distinct_experts(ids)}))
    return 0


def _graph_timed_calls(fn, reps, flush):
    """Median device time (ms) of one CUDA-graph replay of fn() (captured
    once after warm-up), L2 flushed before each replay; None if fn cannot be
    captured."""
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
    except Exception as e:  # capture not possible: report eager only
        print(json.dumps({"graph_capture_error": str(e)[:200]}), file=sys.stderr)
        return None
    return _timed_calls(g.replay, reps, flush)


def run_fp8_peak(local):
    """Burst dense FP8 (e4m3 x e4m3 -> bf16) rate of the vendor library GEMM,
    torch._scaled_mm at 8192^3, best of 10 CUDA-event timings; reported next
    to the roofline denominator (2 x the measured bf16 burst), not used as it."""
    dev = torch.device("cuda", local)
    n = 8192
    g = torch.Generator(device=dev).manual_seed(0)
    a = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device=dev, generator=g).to(torch.float8_e4m3fn)
    one = torch.tensor(1.0, device=dev)
    f = lambda: torch._scaled_mm(a, b.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(3):
        f()
    torch.cuda.synchronize()
    best = None
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        f()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    pk, src = peaks()
    tf = 2.0 * n ** 3 / (best * 1e-3) / 1e12
    print(json.dumps({"fp8_burst_tflops_vendor_gemm": tf, "shape": [n, n, n], "best_ms": best,
                      "bf16_x2_denominator": 2.0 * pk["bf16_tflops"], "bf16_source": src}),
          flush=True)
    return 0


def run_workloads(args, local):
    """One JSON line per shape of the other hot-path configurations (for the
    results tables): per-tensor W8A16, [1,128] block W8A8, fused MoE FP8-block
    and MXFP4.  Each call is timed alone with L2 flushed (a 512 MB read) before it."""
    import mxfp4_quantized_gemm_token_gb300 as mxq
    from mxfp4_quantized_gemm_token_gb300 import synth
    dev = torch.device("cuda", local)
    pk, _ = peaks()
    hbm = pk["hbm_gbs"]
    flush = L2Flush(dev, args.flush)
    reps = args.steps
    names = args.workload.split(",")
    out = []

    def emit(d):
        d["workload"] = name
        print(json.dumps(d), flush=True)

    for name in names:
        if name == "block128":
            # the bench workload per M: the scaled GEMM alone on pre-quantized
            # activations, and the whole linear (quantization + GEMM)
            w, ws = synth.block_fp8_weight(18432, 7168, 128, seed=1, device=dev)
            for M in (1, 8, 17, 128, 1024, 4096):
                x = synth.activations(M, 7168, seed=M, device=dev)
                qa, sa = mxq.per_token_group_quant_fp8(x, 128)
                g = lambda: mxq.fp8_scaled_mm(qa, w, ws, [128, 128], a_scale=sa)
                f = lambda: mxq.w8a8_block_fp8_linear(x, w, [128, 128], ws)
                for _ in range(args.warmup):
                    g()
                    f()
                gemm_ms = _timed_calls(g, reps, flush)
                ms = _timed_calls(f, reps, flush)
                byts = 18432 * 7168 + 144 * 56 * 4 + M * (7168 + 56 * 4) + M * 18432 * 2
                flops = 2 * M * 18432 * 7168
                emit({"M": M, "N": 18432, "K": 7168, "gemm_us": gemm_ms * 1e3, "linear_us": ms * 1e3,
                      "gemm_TFLOPs": flops / gemm_ms / 1e9, "gemm_GBs": byts / gemm_ms / 1e6,
                      "gemm_hbm_frac": byts / gemm_ms / 1e6 / hbm,
                      "gemm_fp8_frac": flops / gemm_ms / 1e9 / (2.0 * pk["bf16_tflops"])})
        elif name == "pertensor":
            a, w, scale, bias = synth.per_tensor_fp8_problem(seed=0)
            a, w, scale, bias = a.to(dev), w.to(dev), scale.to(dev), bias.to(dev)
            for _ in range(args.warmup):
                mxq.fp8_per_tensor_linear(a, w, scale, bias)
            f = lambda: mxq.fp8_per_tensor_linear(a, w, scale, bias)
            ms = _timed_calls(f, reps, flush)
            gms = _graph_timed_calls(f, reps, flush)
            byts = 97 * 576 * 2 + 224 * 576 + 224 * 4 + 97 * 224 * 2
            emit({"M": 97, "N": 224, "K": 576, "us": ms * 1e3,
                  "us_graph": None if gms is None else gms * 1e3,
                  "TFLOPs": 2 * 97 * 224 * 576 / ms / 1e9, "GBs": byts / ms / 1e6})
        elif name == "block1x128":
            w, ws = synth.block_fp8_weight(4096, 7168, 1, seed=1, device=dev)
            for M in (1, 64, 2048):
                if M >= 64:
                    base = synth.activations(M, 7168 + 128, seed=M, device=dev).view(2, M // 2, 7296)
                    x = base[:, :, :7168]
                else:
                    x = synth.activations(M, 7168, seed=M, device=dev)
                f = lambda: mxq.w8a8_block_fp8_linear(x, w, [1, 128], ws)
                qa, sa = mxq.per_token_group_quant_fp8(x, 128)
                qf = lambda: mxq.per_token_group_quant_fp8(x, 128)
                g = lambda: mxq.fp8_scaled_mm(qa, w, ws, [1, 128], a_scale=sa)
                for _ in range(args.warmup):
                    f()
                    g()
                ms = _timed_calls(f, reps, flush)
                gms = _graph_timed_calls(f, reps, flush)
                gemm_ms = _timed_calls(g, reps, flush)
                quant_ms = _timed_calls(qf, reps, flush)
                byts = 4096 * 7168 + 4096 * 56 * 4 + M * 7168 * 2 + M * 4096 * 2
                emit({"M": M, "N": 4096, "K": 7168, "us": ms * 1e3,
                      "us_graph": None if gms is None else gms * 1e3,
                      "gemm_us": gemm_ms * 1e3, "quant_us": quant_ms * 1e3,
                      "TFLOPs": 2 * M * 4096 * 7168 / ms / 1e9, "GBs": byts / ms / 1e6,
                      "hbm_frac": byts / ms / 1e6 / hbm})
        elif name in ("moe_fp8", "moe_mxfp4"):
            fp8 = name == "moe_fp8"
            E, topk, K, N = (256, 8, 7168, 2048) if fp8 else (128, 4, 2880, 2880)
            Ts = (4, 32, 256, 1024) if fp8 else (1, 32, 64, 512)
            if fp8:
                w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=0, device=dev)
                b1 = b2 = None
                per_expert = 2 * N * K + K * N + (s1[0].numel() + s2[0].numel()) * 4
                wt = mxq.W_FP8_BLOCK128
            else:
                w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=0, device=dev)
                b1, b2 = synth.moe_biases(E, N, K, seed=1, device=dev)
                per_expert = (2 * N * K + K * N) // 2 + (2 * N * K + K * N) // 32 + (2 * N + K) * 4
                wt = mxq.W_MXFP4
            for T in Ts:
                for routing in ("uniform", "zipf"):
                    rf = synth.routing_uniform if routing == "uniform" else synth.routing_zipf
                    tw, ids = rf(T, E, topk, seed=T)
                    touched = synth.distinct_experts(ids)
                    x = synth.activations(T, K, seed=T, scale_div=10, device=dev)
                    tw, ids = tw.to(dev), ids.to(dev)
                    bm = args.block_m
                    ws = torch.empty(1, dtype=torch.uint8, device=dev)
                    import ctypes
                    sz = ctypes.c_size_t(0)
                    mxq.check(mxq._lib.load().mxq_fused_experts_workspace_size(
                        T, K, E, N, topk, bm, wt, ctypes.byref(sz)))
                    ws = torch.empty(sz.value, dtype=torch.uint8, device=dev)
                    f = lambda: mxq.fused_experts(x, w1, s1, w2, s2, tw, ids, wtype=wt, w1_bias=b1,
                                                  w2_bias=b2, block_m=bm, workspace=ws)
                    for _ in range(args.warmup):
                        f()
                    mxq.sync_status(dev)
                    ms = _timed_calls(f, reps, flush)
                    gms = _graph_timed_calls(f, reps, flush)
                    byts = touched * per_expert + T * K * 4
                    flops = T * topk * (2 * K * 2 * N + 2 * N * K)
                    bm_used = bm if bm else (32 if T * topk <= 16 * E else 64)
                    emit({"T": T, "routing": routing, "experts_touched": touched, "block_m": bm_used,
                          "us": ms * 1e3, "us_graph": None if gms is None else gms * 1e3, "TFLOPs": flops / ms / 1e9, "GBs": byts / ms / 1e6,
                          "hbm_frac": byts / ms / 1e6 / hbm})
    return 0


def run_ablation(args, local):
    """Per-expert-block path choice vs one path for the whole layer (the global
    crossover, chosen from max(1, S/E)), and both paths forced, on the MoE
    workloads under uniform and Zipf routing.  Threshold SMALL_M_MAX = 16
    slots: blocks (or the layer average) at or below it use the narrowest MMA
    N that covers them, larger ones the full block_m width."""
    import mxfp4_quantized_gemm_token_gb300 as mxq
    from mxfp4_quantized_gemm_token_gb300 import synth, _lib
    dev = torch.device("cuda", local)
    flush = L2Flush(dev, args.flush)
    modes = (("per_block", 0), ("global", 3), ("all_narrow", 1), ("all_full", 2))
    prev = mxq.get_option(_lib.OPT_SMALL_M_MAX)
    try:
        mxq.set_option(_lib.OPT_SMALL_M_MAX, 16)
        for kind in ("fp8", "mxfp4"):
            fp8 = kind == "fp8"
            E, topk, K, N = (256, 8, 7168, 2048) if fp8 else (128, 4, 2880, 2880)
            Ts = (4, 32, 256) if fp8 else (1, 32, 512)
            if fp8:
                w1, s1, w2, s2 = synth.moe_fp8_weights(E, N, K, seed=0, device=dev)
                kw = {}
            else:
                w1, s1, w2, s2 = synth.moe_mxfp4_weights(E, N, K, seed=0, device=dev)
                b1, b2 = synth.moe_biases(E, N, K, seed=1, device=dev)
                kw = dict(wtype=mxq.W_MXFP4, w1_bias=b1, w2_bias=b2)
            for T in Ts:
                for routing in ("uniform", "zipf"):
                    rf = synth.routing_uniform if routing == "uniform" else synth.routing_zipf
                    tw, ids = rf(T, E, topk, seed=T)
                    touched = synth.distinct_experts(ids)
                    x = synth.activations(T, K, seed=T, scale_div=10, device=dev)
                    tw, ids = tw.to(dev), ids.to(dev)
                    line = {"workload": "moe_ablation", "kind": kind, "T": T, "routing": routing,
                            "experts_touched": touched, "avg_m": max(1, T * topk // E),
                            "block_m": args.block_m or (32 if T * topk <= 16 * E else 64),
                            "small_m_max": 16}
                    for name, force in modes:
                        mxq.set_option(_lib.OPT_FORCE_PATH, force)
                        f = lambda: mxq.fused_experts(x, w1, s1, w2, s2, tw, ids,
                                                      block_m=args.block_m, **kw)
                        for _ in range(args.warmup):
                            f()
                        mxq.sync_status(dev)
                        line["us_" + name] = _timed_calls(f, args.steps, flush) * 1e3
                    print(json.dumps(line), flush=True)
    finally:
        mxq.set_option(_lib.OPT_FORCE_PATH, 0)
        mxq.set_option(_lib.OPT_SMALL_M_MAX, prev)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mxq", choices=["mxq", "reference"])
    ap.add_argument("--opt", action="append", default=[],
                    help="library option OPTION=VALUE (MXQ_OPT_* number), repeatable")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--fp8-peak", action="store_true",
                    help="measure the vendor FP8 GEMM burst rate (8192^3) and exit")
    ap.add_argument("--workload", default="",
                    help="comma list of block128, pertensor, block1x128, moe_fp8, moe_mxfp4 (tables only)")
    ap.add_argument("--block-m", type=int, default=0,
                    help="MoE tokens per expert block; 0 = the library's choice")
    ap.add_argument("--profile", type=int, default=0,
                    help="run 3 launches of quant + GEMM at this M only (for ncu)")
    ap.add_argument("--profile-moe", default="",
                    help="kind:T:E, e.g. mxfp4:64:128 -- two fused-MoE calls (for ncu)")
    ap.add_argument("--flush", default="read", choices=["read", "write"],
                    help="L2 flush of the tables: read (default) or write a 512 MB buffer")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu DRAM bytes per launch of the dominant kernel (if measured)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.opt:
        import mxfp4_quantized_gemm_token_gb300 as mxq
        for kv in args.opt:
            k, v = kv.split("=")
            mxq.set_option(int(k), int(v))
    if args.profile:
        return run_profile(args, local)
    if args.fp8_peak:
        return run_fp8_peak(local)
    if args.profile_moe:
        return run_profile_moe(args, local)
    if args.workload == "moe_ablation":
        return run_ablation(args, local)
    if args.workload:
        return run_workloads(args, local)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
