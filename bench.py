"""Benchmark of the block-FP8 MoE layer forward on GB300.

Workload (default): the largest single-GPU layer the metric is quoted on -- 32 experts, hidden
7168, intermediate 2048, top-8, FP8 E4M3 weights with 128x128 UE8M0 (power-of-two) block scales,
UE8M0 1x128 activation scales, BF16 activations, softmax top-8 routing -- at a token capacity of
4096 with all 4096 tokens live.  The same run also measures ("sweep") the decode layer (288 experts,
hidden 4096, intermediate 512, SwiGLU clamped at 7.0, FP32 scales) at M = 1, 4 and 32, the padded
layer at capacity 512 with 16 live tokens, and the padded layer with FP32 weight and activation
scales at 512/16 and 4096/4096.  One step = one full layer forward (routing alignment, activation
quantization, FC1 + SwiGLU + requant, FC2, top-k reduce) replayed from a CUDA graph, with L2 flushed
(a 512 MB write, larger than the 129 MB L2) before every step; the step time is taken with CUDA
events around the replay on the launching stream.

Prints one JSON line.  `--impl reference` times the CPU oracle on the host cores instead (the
reference arm).  `--measure-peaks` times the dense FP8 GEMM peak (torch._scaled_mm, e4m3 8192^3).
Under torchrun every rank runs its own replica of the layer on its own batch (weak scaling: the
layer has no exchange step between data-parallel replicas); rank 0 prints the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer us and % of FP8/HBM roofline vs live tokens M (1 GB300)"
WORKLOAD = "padded"
# (workload, token capacity, live tokens) measured beside the headline point
SWEEP_POINTS = (("decode", 1, 1), ("decode", 4, 4), ("decode", 32, 32), ("padded", 512, 16),
                ("padded_fp32", 512, 16), ("padded_fp32", 4096, 4096))
KERNELS = ("align", "quant", "fc1", "fc2", "reduce")
FLUSH_BYTES = 512 << 20


# ------------------------------------------------------------------ peaks
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def fp8_peak(peaks):
    """Dense FP8 GEMM peak in TFLOP/s and where it comes from: the cuBLASLt e4m3 GEMM measured on this
    part (profiles/fp8_peak.json, written from `bench.py --measure-peaks`), else twice the measured
    BF16 peak (nominal 4.5 vs 2.25 PFLOP/s)."""
    try:
        with open(os.path.join(ROOT, "profiles", "fp8_peak.json")) as f:
            rec = json.load(f)
        return float(rec["fp8_tflops"]), "measured: torch._scaled_mm e4m3 8192^3, best of 10 (profiles/fp8_peak.json)"
    except (OSError, KeyError, ValueError):
        return 2.0 * peaks["bf16_tflops"], f"{peaks['source']}: 2 x MEASURED_PEAKS bf16_tflops"


# ------------------------------------------------------- algorithmic work
def layer_work(case: synth.LayerCase):
    """Algorithmic FLOPs and bytes of one layer forward and of its FC1 launch.

    Layer bytes: weights (codes + block scales) of the occupied experts only, x in and out in
    BF16, ids and routing weights; intermediates are not counted.  FC1 launch bytes: the occupied
    experts' W13 codes + scales, the FP8 activation rows and scales it reads, and the FC2-input
    codes and scales it writes.
    """
    sh = case.shape
    ids = case.topk_ids[: case.n]
    valid = ids[(ids >= 0) & (ids < sh.E)]
    occ = int(np.unique(valid).size)
    P = int(valid.size)
    H, I = sh.H, sh.I
    sc = 1 if sh.weight_fmt == synth.SCALE_UE8M0 else 4
    asc = 1 if sh.act_fmt == synth.SCALE_UE8M0 else 4
    w13_bytes = 2 * I * H + sc * (2 * I // 128) * (H // 128)
    w2_bytes = H * I + sc * (H // 128) * (I // 128)
    return {
        "occupied_experts": occ, "pairs": P,
        "flops": 6.0 * P * H * I,
        "layer_bytes": occ * (w13_bytes + w2_bytes) + 4 * case.n * H + 8 * case.n * sh.topk,
        "fc1_bytes": occ * w13_bytes + P * (H + asc * H // 128) + P * (I + asc * I // 128),
        "fc1_flops": 4.0 * P * H * I,
    }


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of the SM clock and throttle reasons while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# ------------------------------------------------------------- ncu traffic
def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "block_fp8_mixture_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(key: str):
    """DRAM bytes per launch from the committed ncu summary, when it was taken on these sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(key)
    if not entry or entry.get("source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


FMT_NAMES = {0: "fp32", 1: "fp32-pow2", 2: "ue8m0"}


def launches_per_forward(case: synth.LayerCase) -> int:
    """Kernels one layer forward launches: alignment (plus its per-CTA counting kernel when the
    plan aligns with several CTAs), quantization, FC1, the SwiGLU + requantization kernel of the
    FP32-scale tile schedule, FC2 and the top-k reduction."""
    import block_fp8_mixture_gb300 as moe
    sh = case.shape
    plan = moe.workspace_plan(case.M_cap, sh.E, sh.H, sh.I, sh.topk, sh.act_fmt)
    block_scaled = sh.weight_fmt == synth.SCALE_UE8M0 and sh.act_fmt == synth.SCALE_UE8M0
    split_swiglu = plan["small_batch"] == 0 and plan["g1"] != 0 and not block_scaled
    return 5 + (plan["align_ctas"] > 1) + split_swiglu


def workload_name(shape, M, n):
    live = f"M={M}" if n == M else f"capacity {M}, {n} live"
    return f"{shape.name} MoE layer E={shape.E} H={shape.H} I={shape.I} top-{shape.topk} {live}"


def bench_config(shape, M, n, world):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": workload_name(shape, M, n),
            "clamp": ("none" if shape.clamp_mode == 0 else
                      f"SwiGLU clamp {shape.limit} {'before' if shape.clamp_mode == 1 else 'after'} SiLU"),
            "scales": f"weights {FMT_NAMES[shape.weight_fmt]} 128x128, activations {FMT_NAMES[shape.act_fmt]} 1x128",
            "l2": "flushed before every step (512 MB write)", "timing": "CUDA graph replay, CUDA events",
            "parallelism": f"replicas x{world}"}


def point_key(workload, M, n):
    return f"{workload} {M}" if n == M else f"{workload} {M}/{n}"


# ------------------------------------------------------------ our arm
class LayerBench:
    def __init__(self, workload, M, n, rank, weights, dev_weights):
        import torch
        import block_fp8_mixture_gb300 as moe
        self.moe = moe
        self.M = M
        self.case = synth.make_case(workload, M, n, seed=2000 + M + 7919 * rank, weights=weights)
        sh = self.case.shape
        self.sh = sh
        self.x = torch.from_numpy(self.case.x_bits.view(np.int16)).cuda().view(torch.bfloat16)
        self.ids = torch.from_numpy(self.case.topk_ids).cuda()
        self.wts = torch.from_numpy(self.case.topk_weights).cuda()
        self.w13, self.s13, self.w2, self.s2 = dev_weights
        self.layer = moe.MoELayer(self.w13, self.s13, self.w2, self.s2, weight_fmt=sh.weight_fmt,
                                  act_fmt=sh.act_fmt, clamp_mode=sh.clamp_mode,
                                  clamp_limit=sh.limit, max_tokens=M, topk=sh.topk)
        self.out = torch.empty((M, sh.H), dtype=torch.bfloat16, device="cuda")
        self.d_n = torch.tensor([self.case.n], dtype=torch.int32, device="cuda")
        self.args = self.layer.args(self.x, self.ids, self.wts, self.out, d_num_tokens=self.d_n)
        self.ws = self.layer.workspace

    def forward(self, stream):
        self.moe.forward(self.args, self.ws, stream)

    def steps(self, stream):
        """The five steps as separate C-ABI calls (same kernels as forward())."""
        moe, sh, ws = self.moe, self.sh, self.ws
        return [
            lambda: moe.align(self.ids, sh.E, sh.H, sh.I, ws, d_num_tokens=self.d_n, act_fmt=sh.act_fmt,
                              stream=stream),
            lambda: moe.quant_act(self.x, sh.topk, sh.E, sh.I, ws, d_num_tokens=self.d_n,
                                  act_fmt=sh.act_fmt, stream=stream),
            lambda: moe.fc1_swiglu_quant(self.args, ws, stream),
            lambda: moe.fc2(self.args, ws, stream),
            lambda: moe.topk_reduce(self.args, ws, stream),
        ]


def run_ours(args, rank, world):
    import torch
    import block_fp8_mixture_gb300 as moe

    moe.load_library()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    peaks = load_peaks()
    fp8_tflops, fp8_source = fp8_peak(peaks)
    hbm_peak = peaks["hbm_gbs"]
    head = (args.workload, args.M, args.n)
    do_sweep = not (args.no_sweep or args.profile_run)
    if not do_sweep:
        points = [head]
    elif args.sweep:
        points = [(args.workload, m, n) for m, n in synth.SWEEPS[args.workload]]
    elif args.workload == WORKLOAD:
        points = list(SWEEP_POINTS)
    else:
        points = []
    points = [head] + [pt for pt in points if pt != head]

    weights, dev_w = {}, {}
    for wl, _, _ in points:
        if wl not in weights:
            weights[wl] = synth.make_weights(synth.SHAPES[wl])
            dev_w[wl] = tuple(torch.from_numpy(a).cuda() for a in
                              (weights[wl].w13, weights[wl].s13, weights[wl].w2, weights[wl].s2))
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    benches = {pt: LayerBench(pt[0], pt[1], pt[2], rank, weights[pt[0]], dev_w[pt[0]]) for pt in points}

    # graphs of the whole forward, one per point
    graphs = {}
    with torch.cuda.stream(stream):
        for pt, b in benches.items():
            b.forward(stream)
            stream.synchronize()
            assert moe.last_device_status(b.ws, stream) == moe.MOE_OK
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                b.forward(stream)
            graphs[pt] = g
    torch.cuda.synchronize()

    def timed_graph(pt, steps, warmup):
        g = graphs[pt]
        times = []
        with torch.cuda.stream(stream):
            for i in range(warmup + steps):
                flush.fill_(i & 0xFF)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                if i >= warmup:
                    times.append((e0, e1))
        stream.synchronize()
        return [a.elapsed_time(b) * 1e3 for a, b in times]   # us

    def per_kernel(pt, steps):
        b = benches[pt]
        fns = b.steps(stream)
        acc = {k: [] for k in KERNELS}
        with torch.cuda.stream(stream):
            for i in range(steps + 2):
                flush.fill_(i & 0xFF)
                if hasattr(torch.cuda, "_sleep"):
                    torch.cuda._sleep(2_000_000)   # let the host queue the launches ahead
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(fns) + 1)]
                evs[0].record(stream)
                for f, e in zip(fns, evs[1:]):
                    f()
                    e.record(stream)
                stream.synchronize()
                if i >= 2:
                    for k, a, c in zip(KERNELS, evs[:-1], evs[1:]):
                        acc[k].append(a.elapsed_time(c) * 1e3)
        return {k: statistics.mean(v) for k, v in acc.items()}

    def e2e(pt, steps, warmup):
        """The layer through the public API with every step's inputs copied in from pinned host
        memory and its output copied back, pipelined the way a caller running many forwards would
        run them: two staging slots, the input copy of step i+1 and the output copy of step i on
        their own streams, overlapping the compute of steps i and i+1.  The span from the first
        input copy to the last output copy, divided by the step count, is the time per step."""
        b = benches[pt]
        parts = [b.x, b.ids, b.wts]
        offs, size = [], 0
        for t in parts:
            offs.append(size)
            size += (t.numel() * t.element_size() + 255) // 256 * 256
        slots = []
        for _ in range(2):
            stage_h = torch.empty(size, dtype=torch.uint8).pin_memory()
            stage_d = torch.empty(size, dtype=torch.uint8, device="cuda")
            views_d = []
            for t, o in zip(parts, offs):
                nb = t.numel() * t.element_size()
                stage_h[o:o + nb].view(t.dtype).view(t.shape).copy_(t.cpu())
                views_d.append(stage_d[o:o + nb].view(t.dtype).view(t.shape))
            out_h = torch.empty(b.out.shape, dtype=b.out.dtype).pin_memory()
            out_d = torch.empty_like(b.out)
            slots.append({"stage_h": stage_h, "stage_d": stage_d, "views": views_d, "out_h": out_h,
                          "out_d": out_d})
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event(enable_timing=False)   # noqa: E731

        def run(n):
            done_compute, done_d2h = [None, None], [None, None]
            for i in range(n):
                sl = slots[i % 2]
                with torch.cuda.stream(h2d_s):
                    if done_compute[i % 2] is not None:
                        h2d_s.wait_event(done_compute[i % 2])   # step i-2 has read this slot
                    sl["stage_d"].copy_(sl["stage_h"], non_blocking=True)
                    in_ready = ev()
                    in_ready.record(h2d_s)
                stream.wait_event(in_ready)
                if done_d2h[i % 2] is not None:
                    stream.wait_event(done_d2h[i % 2])          # step i-2's output was copied out
                x_d, ids_d, w_d = sl["views"]
                b.layer(x_d, ids_d, w_d, out=sl["out_d"], stream=stream)
                done_compute[i % 2] = ev()
                done_compute[i % 2].record(stream)
                with torch.cuda.stream(d2h_s):
                    d2h_s.wait_event(done_compute[i % 2])
                    sl["out_h"].copy_(sl["out_d"], non_blocking=True)
                    done_d2h[i % 2] = ev()
                    done_d2h[i % 2].record(d2h_s)

        run(warmup)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(h2d_s)
        run(steps)
        e1.record(d2h_s)          # after the last output copy (which follows the last compute)
        torch.cuda.synchronize()
        h2d = slots[0]["stage_h"].numel()
        d2h = slots[0]["out_h"].numel() * slots[0]["out_h"].element_size()
        return e0.elapsed_time(e1) * 1e3 / steps, h2d, d2h

    if args.profile_run:
        us = timed_graph(head, args.steps, args.warmup)
        return {"profile_run": True, "point": point_key(*head), "us_mean": statistics.mean(us)}

    # pre-warm (clocks settle), then the timed region of the headline point
    clock = ClockSampler(torch.cuda.current_device())
    t_end = time.time() + 0.5
    while time.time() < t_end:
        timed_graph(head, 5, 0)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    us = timed_graph(head, args.steps, args.warmup)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    wall = time.perf_counter() - t0
    clocks = clock.stop()

    us_mean = statistics.mean(us)
    if dist is not None:
        t = torch.tensor([us_mean], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        us_mean = float(t.item())

    work = layer_work(benches[head].case)
    kern = per_kernel(head, max(10, min(args.steps, 50)))
    fc1_us = kern["fc1"]
    traffic = ncu_traffic(f"fc1_{args.workload}_M{args.M}")
    sched = "block-scaled 128-row tiles" if (benches[head].sh.weight_fmt == synth.SCALE_UE8M0 and
                                             benches[head].sh.act_fmt == synth.SCALE_UE8M0) else "FC1 schedule"
    if work["fc1_flops"] / (fp8_tflops * 1e12) > work["fc1_bytes"] / (hbm_peak * 1e9):
        achieved = work["fc1_flops"] / (fc1_us * 1e-6) / 1e12
        roofline = {"kernel": f"fc1 (grouped GEMM + SwiGLU + requant, {sched})", "bound": "tensor",
                    "achieved": achieved, "peak": fp8_tflops, "unit": "TFLOP/s",
                    "frac": achieved / fp8_tflops, "traffic": traffic,
                    "algorithmic_flops": work["fc1_flops"], "avg_launch_us": fc1_us,
                    "peak_source": fp8_source}
    else:
        achieved = work["fc1_bytes"] / (fc1_us * 1e-6) / 1e9
        roofline = {"kernel": "fc1 (grouped GEMM + SwiGLU + requant)", "bound": "hbm",
                    "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": traffic,
                    "algorithmic_bytes": work["fc1_bytes"], "avg_launch_us": fc1_us,
                    "peak_source": f"{peaks['source']} (MEASURED_PEAKS hbm_gbs)"}

    def layer_roof(pt, t_us):
        w = layer_work(benches[pt].case)
        t_f = w["flops"] / (fp8_tflops * 1e12)
        t_b = w["layer_bytes"] / (hbm_peak * 1e9)
        return {"us": t_us, "roofline_us": max(t_f, t_b) * 1e6,
                "frac_of_roofline": max(t_f, t_b) * 1e6 / t_us,
                "bound": "tensor" if t_f > t_b else "hbm",
                "tflops": w["flops"] / (t_us * 1e-6) / 1e12,
                "gbs": w["layer_bytes"] / (t_us * 1e-6) / 1e9,
                "occupied_experts": w["occupied_experts"]}

    sweep_out = {}
    for pt in points:
        steps_us = us if pt == head else timed_graph(pt, max(20, args.steps // 2), 3)
        t_us = us_mean if pt == head else statistics.mean(steps_us)
        key = point_key(*pt)
        sweep_out[key] = layer_roof(pt, t_us)
        sweep_out[key]["p50_us"] = statistics.median(steps_us)
        sweep_out[key]["per_kernel_us"] = kern if pt == head else per_kernel(pt, 20)

    e2e_us, h2d, d2h = e2e(head, max(10, min(args.steps, 100)), 3)

    shape = synth.SHAPES[args.workload]
    line = {
        "metric": METRIC, "value": us_mean, "unit": "us", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": us_mean / 1e3, "higher_is_better": False,
        "p50_us": statistics.median(us),
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
        "config": bench_config(shape, args.M, args.n, world),
        "roofline": roofline,
        "layer_roofline": sweep_out[point_key(*head)],
        "fp8_peak_tflops": fp8_tflops, "fp8_peak_source": fp8_source,
        "sweep": sweep_out,
        "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "MoELayer.__call__ (C ABI moe_fp8_block_forward); every step copies its x, "
                       "ids and routing weights in from a pinned staging buffer and its output "
                       "back to pinned memory; steps pipelined over two staging slots with the "
                       "copies on their own streams; no L2 flush (the 1.4 GB of weights exceed L2)",
                "pipelined": True},
        "gpu_launches": launches_per_forward(benches[head].case) * args.steps,
        "clocks": clocks,
        "timed_wall_s": wall,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(benches[head].case)
    if dist is not None:
        dist.destroy_process_group()
    return line


# ------------------------------------------------------------ FP8 peak
def measure_peaks():
    """Dense FP8 GEMM throughput of this part: torch._scaled_mm (cuBLASLt) on e4m3 8192^3 with
    per-tensor scales and a BF16 output, best of 10 (burst) and back to back for 4 s (sustained), with
    the SM clocks sampled meanwhile."""
    import torch
    n = 8192
    flops = 2.0 * n ** 3
    a = (torch.randn(n, n, device="cuda") * 0.5).to(torch.float8_e4m3fn)
    b = (torch.randn(n, n, device="cuda") * 0.5).to(torch.float8_e4m3fn).t()   # column-major
    one = torch.ones((), device="cuda", dtype=torch.float32)

    def mm():
        return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

    for _ in range(5):
        mm()
    torch.cuda.synchronize()
    clock = ClockSampler(torch.cuda.current_device())
    best = float("inf")
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e-3)
    t_end = time.time() + 4.0
    reps, e0 = 0, torch.cuda.Event(enable_timing=True)
    e0.record()
    while time.time() < t_end:
        for _ in range(20):
            mm()
        reps += 20
        torch.cuda.synchronize()
    e1 = torch.cuda.Event(enable_timing=True)
    e1.record()
    e1.synchronize()
    sustained = flops * reps / (e0.elapsed_time(e1) * 1e-3) / 1e12
    return {"fp8_tflops": flops / best / 1e12, "fp8_tflops_sustained": sustained,
            "how": "torch._scaled_mm float8_e4m3fn 8192^3 (2 N^3 flops), per-tensor scales, bf16 out: "
                   "best of 10 (burst); back to back for 4 s (sustained); CUDA events",
            "torch": torch.__version__, "gpu": torch.cuda.get_device_name(),
            "clocks": clock.stop()}


# ---------------------------------------------------------- the oracle arm
def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_tokens(case: synth.LayerCase, tokens):
    import oracle
    sh, w = case.shape, case.weights
    return oracle.moe_forward(case.x, case.topk_ids, case.topk_weights, w.w13, w.s13, w.w2, w.s2,
                              act_fmt=sh.act_fmt, weight_fmt=sh.weight_fmt,
                              clamp_mode=sh.clamp_mode, limit=sh.limit, tokens=tokens)


def time_oracle(case: synth.LayerCase, budget_s: float, max_tokens=None):
    """Seconds per token of the oracle (as it stands), timed token by token on a sample of the
    case's tokens until about budget_s has been spent."""
    order = np.random.default_rng(0).permutation(case.n)
    limit = case.n if max_tokens is None else min(case.n, max_tokens)
    done, spent = 0, 0.0
    while done < limit and (spent < budget_s or done == 0):
        t0 = time.perf_counter()
        oracle_tokens(case, order[done: done + 1])
        spent += time.perf_counter() - t0
        done += 1
    return spent / done, done


def cpu_baseline(case: synth.LayerCase, budget_s: float = 12.0):
    sec_tok, done = time_oracle(case, budget_s)
    us_layer = sec_tok * case.n * 1e6
    return {"value": us_layer, "unit": "us", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{done} of the {case.n} tokens of the same layer, one at a time, "
                      f"time per token x {case.n} (numpy, BLAS default threads)"}


def reference_arm(args):
    """The oracle on this arm's config: each step sends one of the live tokens (a different one
    per step) through it. ms_per_step is that step's wall time; value scales the mean step time to
    the whole layer (x live tokens)."""
    shape = synth.SHAPES[args.workload]
    weights = synth.make_weights(shape)
    case = synth.make_case(args.workload, args.M, args.n, seed=2000 + args.M, weights=weights)
    order = np.random.default_rng(0).permutation(case.n)
    per_step = []
    for i in range(args.warmup + args.steps):
        j = i % case.n
        t0 = time.perf_counter()
        oracle_tokens(case, order[j: j + 1])
        per_step.append(time.perf_counter() - t0)
    sec_step = statistics.mean(per_step[args.warmup:])
    us_layer = sec_step * case.n * 1e6
    return {
        "impl": "reference", "metric": METRIC, "value": us_layer, "unit": "us",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec_step * 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3", "data": "synthetic",
        "config": bench_config(shape, args.M, args.n, 1),
        "cpu_baseline": {"value": us_layer, "unit": "us", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: 1 of the {case.n} live tokens of the same layer "
                                   f"through the oracle (a different token per step); ms_per_step "
                                   f"is that step's wall time, value = mean step time x {case.n}"},
        "e2e": {"value": us_layer, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(synth.SHAPES),
                    help="layer shape (default: the padded layer E=32 H=7168 I=2048)")
    ap.add_argument("--M", type=int, default=None, help="token capacity of the headline point")
    ap.add_argument("--n", type=int, default=None,
                    help="live tokens at --M (default: the workload's live count for M, else M)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="measure every point of --workload's sweep (default: the fixed list of "
                         "points beside the default workload)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-run", action="store_true",
                    help="only W + K graph replays of the headline point (for ncu captures)")
    ap.add_argument("--measure-peaks", action="store_true",
                    help="time the dense FP8 GEMM peak and print it as JSON")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    if args.M is None:
        args.M = {"decode": 32, "tiny": 16}.get(args.workload, 4096)
    if args.n is None:   # the workload's live count at this capacity (16 of 512 for padded)
        args.n = dict(synth.SWEEPS.get(args.workload, [])).get(args.M, args.M)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.measure_peaks:
        print(json.dumps(measure_peaks()), flush=True)
        return 0
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return 0
    line = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
