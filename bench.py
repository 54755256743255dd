"""Benchmark of the FP8 delayed-scaling path on GB300.

One step is the FP8 bookkeeping of one MLP training step on the FFN workload
(sequence 2048 x batch 4, hidden 4096, FFN 16384, bf16):

  1. fp8q_quantize_amax        activation 8192x16384 bf16 -> e4m3fn + amax
  2. fp8q_multi_quantize_amax  W1 4096x16384 and W2 16384x4096 -> e4m3fn, one launch
  3. fp8q_dequantize           e5m2 gradient 8192x16384 -> bf16
  4. fp8q_amax_scale_update    96 layers x 6 slots, history 1024 -> next step's scales

Step 4 reads the amaxes steps 1-2 wrote and writes the scales steps 1-3 read
on the next step (delayed scaling entirely on the device).  Inputs are
seeded synthetic tensors resident in HBM; each step streams ~1.2 GB, far more
than the 129 MB L2, so no input is L2-resident when it is read again.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "quantize+amax HBM GB/s (% of GB300 peak); scale-update µs per 576-slot call"
WORKLOAD = ("FP8 delayed-scaling step, FFN config: quantize+amax act 8192x16384 e4m3fn; W1 4096x16384 + "
            "W2 16384x4096 e4m3fn in one multi-tensor launch; dequantize grad 8192x16384 e5m2; "
            "update 576 slots x 1024")

ACT = (8192, 16384)
W1 = (4096, 16384)
W2 = (16384, 4096)
GRAD = (8192, 16384)
H, S = 1024, 576

N_ACT = ACT[0] * ACT[1]
N_W = W1[0] * W1[1] + W2[0] * W2[1]
N_GRAD = GRAD[0] * GRAD[1]
BYTES_PER_ELEM = 3                      # 2 B bf16 read + 1 B fp8 written (or the reverse)
UPDATE_BYTES = 2 * H * S * 4 + S * 4 + 4 * S * 4   # history read+write, amax_new, scale & scale_inv r+w
BYTES_QUANT = BYTES_PER_ELEM * N_ACT
BYTES_MULTI = BYTES_PER_ELEM * N_W
BYTES_DEQ = BYTES_PER_ELEM * N_GRAD
STEP_BYTES = BYTES_QUANT + BYTES_MULTI + BYTES_DEQ + UPDATE_BYTES
KERNELS_PER_STEP = 4


# --------------------------------------------------------------------------- peaks and clocks

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """Reads SM clock, max clock, power and clock-event reasons through NVML.

    Only reads device state; never changes a setting.
    """
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, torch_device_index: int):
        self.ok = False
        self.samples = []
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            import torch
            uuid = getattr(torch.cuda.get_device_properties(torch_device_index), "uuid", None)
            rc = 1
            if uuid is not None:
                rc = self.nv.nvmlDeviceGetHandleByUUID(("GPU-" + str(uuid)).encode(), ctypes.byref(self.h))
            if rc != 0:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
                idx = int(vis.split(",")[torch_device_index]) if vis and vis.split(",")[0].isdigit() \
                    else torch_device_index
                rc = self.nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.h))
            if rc != 0:
                return
            self._reasons = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            rc = self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = mx.value if rc == 0 else None
            self.ok = True
        except OSError:
            self.ok = False

    def sample(self):
        if not self.ok:
            return
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        p = ctypes.c_uint()
        if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) != 0:
            return
        self._reasons(self.h, ctypes.byref(r))
        self.nv.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(p))
        self.samples.append((c.value, r.value, p.value / 1000.0))

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": getattr(self, "max_mhz", None), "reasons": [],
                    "samples": 0, "source": "nvml" if self.ok else "unavailable"}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for s in self.samples:
            bits |= s[1]
        reasons = [name for b, name in self.REASONS.items() if bits & b and name != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "power_w_max": max(s[2] for s in self.samples),
                "source": "nvml on the host, during the timed steps"}


# --------------------------------------------------------------------------- multi-rank helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, group=None) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend(group) == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate_throughput(bytes_per_rank: float, seconds_per_rank: float, world_size: int, group=None):
    """Whole-job GB/s: bytes all ranks processed over the slowest rank's time."""
    t = max_over_ranks(seconds_per_rank, group)
    return bytes_per_rank * world_size / t / 1e9, t


# --------------------------------------------------------------------------- workload

class Step:
    """Device-resident state of one benchmark step."""

    def __init__(self, dev):
        import torch
        from quantize_amax_scaling_gb300 import fp8q
        from quantize_amax_scaling_gb300 import workloads as W
        self.fp8q = fp8q
        self.dev = dev
        self.act = W.gelu_activation(W.SEED_FFN, dev).reshape(-1)
        ffn = W.ffn_tensors(dev)
        self.w = [ffn[1].reshape(-1), ffn[2].reshape(-1)]
        del ffn
        grad = W.gradient(GRAD, W.SEED_GRAD, dev).reshape(-1)
        hist, new, scale, scale_inv, slot_format = W.scale_update_inputs(dev)
        self.hist, self.amax_new, self.slot_format = hist, new, slot_format
        self.scale, self.scale_inv = scale, scale_inv
        # realistic starting scales: one update from the synthetic amaxes
        fp8q.fp8q_amax_scale_update(self.hist, self.amax_new, self.scale, self.scale_inv,
                                    fp8q.E4M3FN, fp8q.ALGO_MAX, 0, self.slot_format)
        # the gradient arrives already in e5m2 (quantized once with its own slot)
        self.grad_q = torch.empty(grad.numel(), dtype=torch.uint8, device=dev)
        gam = torch.zeros(1, device=dev)
        fp8q.fp8q_quantize_amax(grad, self.grad_q, fp8q.E5M2, self.scale[4:5], gam)
        del grad
        self.q_act = torch.empty(self.act.numel(), dtype=torch.uint8, device=dev)
        self.q_w = [torch.empty(w.numel(), dtype=torch.uint8, device=dev) for w in self.w]
        self.y_grad = torch.empty(self.grad_q.numel(), dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize(dev)

    def run(self, stream, events=None):
        """Enqueue one step on `stream`; `events` (5 CUDA events) bracket the four kernels."""
        f = self.fp8q
        st = stream.cuda_stream
        self.amax_new[:3].zero_()  # this step's amax slots start from 0 (max-accumulated)
        if events:
            events[0].record(stream)
        f.fp8q_quantize_amax(self.act, self.q_act, f.E4M3FN, self.scale[0:1], self.amax_new[0:1], st)
        if events:
            events[1].record(stream)
        f.fp8q_multi_quantize_amax(self.w, self.q_w, f.E4M3FN, [self.scale[1:2], self.scale[2:3]],
                                   [self.amax_new[1:2], self.amax_new[2:3]], st)
        if events:
            events[2].record(stream)
        f.fp8q_dequantize(self.grad_q, self.y_grad, f.E5M2, self.scale[4:5], st)
        if events:
            events[3].record(stream)
        f.fp8q_amax_scale_update(self.hist, self.amax_new, self.scale, self.scale_inv, f.E4M3FN,
                                 f.ALGO_MAX, 0, self.slot_format, st)
        if events:
            events[4].record(stream)


    def run_branched(self, stream, side):
        """The same step for graph capture, with the three streaming kernels on parallel
        branches (they touch disjoint tensors): forked after the amax reset, joined before
        the update that reads their amaxes, so one kernel's ramp and tail overlap another's."""
        import torch
        f = self.fp8q
        self.amax_new[:3].zero_()
        fork = torch.cuda.Event()
        fork.record(stream)
        for s in side:
            s.wait_event(fork)
        f.fp8q_quantize_amax(self.act, self.q_act, f.E4M3FN, self.scale[0:1], self.amax_new[0:1],
                             stream.cuda_stream)
        f.fp8q_multi_quantize_amax(self.w, self.q_w, f.E4M3FN, [self.scale[1:2], self.scale[2:3]],
                                   [self.amax_new[1:2], self.amax_new[2:3]], side[0].cuda_stream)
        f.fp8q_dequantize(self.grad_q, self.y_grad, f.E5M2, self.scale[4:5], side[1].cuda_stream)
        for s in side:
            join = torch.cuda.Event()
            join.record(s)
            stream.wait_event(join)
        f.fp8q_amax_scale_update(self.hist, self.amax_new, self.scale, self.scale_inv, f.E4M3FN,
                                 f.ALGO_MAX, 0, self.slot_format, stream.cuda_stream)


def run_gpu(args, ws, rank, local):
    import torch
    import torch.distributed as dist
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    step = Step(dev)
    stream = torch.cuda.Stream(dev)
    peak, peak_src = measured_peaks()
    torch.cuda.synchronize(dev)  # the step's inputs, made on the default stream, are complete

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step.run(stream)
    torch.cuda.synchronize(dev)

    # The step is captured as CUDA graphs (its four library kernels and the
    # amax reset): one graph of G consecutive steps and one of a single step,
    # replayed so that exactly K steps run, with no host launches between them.
    # Within a step the three streaming kernels are parallel branches joined
    # before the update (run_branched); steps follow one another in order.
    G = max(1, min(args.steps, 10))
    side = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]
    graph_g, graph_1 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph_g, stream=stream):
            for _ in range(G):
                step.run_branched(stream, side)
        with torch.cuda.graph(graph_1, stream=stream):
            step.run_branched(stream, side)
        for _ in range(args.warmup):
            graph_1.replay()
        graph_g.replay()
    torch.cuda.synchronize(dev)

    # ---- timed region: K graph replays back to back, CUDA events only at its two ends
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps // G):
            graph_g.replay()
        for _ in range(args.steps % G):
            graph_1.replay()
        end.record(stream)
    while not end.query():          # sample clocks while the GPU runs the timed steps
        clocks.sample()
        time.sleep(0.002)
    torch.cuda.synchronize(dev)
    barrier()
    t_rank = start.elapsed_time(end) / 1e3          # seconds for all K steps on this rank
    value, t_max = aggregate_throughput(STEP_BYTES * args.steps, t_rank, ws)

    # ---- the same K steps launched kernel by kernel from the host (eager)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e_start.record(stream)
        for _ in range(args.steps):
            step.run(stream)
        e_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    eager_value, eager_t = aggregate_throughput(STEP_BYTES * args.steps, e_start.elapsed_time(e_end) / 1e3, ws)

    # ---- the same K steps again with an event around every kernel, for the
    # per-kernel breakdown and the roofline.  An event between two kernels
    # keeps the second from overlapping the first one's tail, so these times
    # are a little longer than the kernels' share of the clean region above.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for k in range(args.steps):
            step.run(stream, ev[k])
    torch.cuda.synchronize(dev)
    barrier()

    per = {"quantize_amax": [], "multi_quantize_amax": [], "dequantize": [], "amax_scale_update": []}
    for k in range(args.steps):
        e = ev[k]
        for j, name in enumerate(per):
            per[name].append(e[j].elapsed_time(e[j + 1]) * 1e3)  # us
    avg = {n: sum(v) / len(v) for n, v in per.items()}
    kbytes = {"quantize_amax": BYTES_QUANT, "multi_quantize_amax": BYTES_MULTI,
              "dequantize": BYTES_DEQ, "amax_scale_update": UPDATE_BYTES}
    kernels = {n: {"us": round(avg[n], 3), "us_median": round(statistics.median(per[n]), 3),
                   "GB/s": round(kbytes[n] / (avg[n] * 1e-6) / 1e9, 1),
                   "frac_of_peak": round(kbytes[n] / (avg[n] * 1e-6) / 1e9 / peak, 4)}
               for n in per}
    q_gbs = kbytes["quantize_amax"] / (avg["quantize_amax"] * 1e-6) / 1e9

    # ---- the same step as one CUDA graph (no host launches, no events inside)
    graph = None if args.no_extras else measure_graph(args, step, stream, dev)

    # ---- rows beyond the step (fused Q->DQ, ring history), timed on their own after it
    next_rows = None if args.no_extras else measure_next_rows(args, step, stream, dev, peak)

    # ---- the other quantize workloads: MLP activation (L2 flushed) and the ragged list
    other_configs = None if args.no_extras else measure_other_configs(step, stream, dev, peak)

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, step, stream, dev) if not args.no_e2e else None

    if rank != 0:
        return None
    traffic = read_traffic()
    upd_graph = graph["scale_update_us_after_dequantize"] if graph else None
    detail = {
        "eager": {"value": round(eager_value, 1), "unit": "GB/s", "ms_per_step": round(eager_t / args.steps * 1e3, 4)},
        "kernels": kernels, "graph": graph, "next_rows": next_rows, "other_configs": other_configs, "e2e": e2e,
        "timing": "value and ms_per_step: K steps replayed from CUDA graphs (10 steps per graph, plus single-step "
                  "replays for a remainder; in each step quantize, multi-tensor quantize and dequantize are "
                  "parallel branches joined before the update), CUDA events only around the region; eager: the "
                  "same K steps launched kernel by kernel; kernels and roofline: a third pass of K eager steps "
                  "with an event around each kernel",
    }
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; FFN/MLP and 96-layer shapes)",
        "config": {"workload": WORKLOAD, "step_bytes": STEP_BYTES,
                   "l2": "inputs larger than L2 (a step streams 1.21 GB)",
                   "parallelism": f"replicas x{ws} (no collective)"},
        # the metric's two halves: the quantize+amax kernel on the 8192x16384
        # activation, and the 576-slot update's device time (CUDA graphs)
        "quantize_amax_gbs": round(q_gbs, 1),
        "quantize_amax_frac": round(q_gbs / peak, 4),
        "scale_update_us": upd_graph if upd_graph is not None else round(avg["amax_scale_update"], 3),
        "scale_update_us_eager": round(avg["amax_scale_update"], 3),
        "scale_update_launches": 1,
        # what a one-element torch fill costs in the update's place in the same graphs
        "graph_node_floor_us": graph["one_element_fill_us_after_dequantize"] if graph else None,
        "roofline": {"kernel": "quantize_amax_kernel 8192x16384", "bound": "hbm", "achieved": round(q_gbs, 1),
                     "peak": peak, "unit": "GB/s", "frac": round(q_gbs / peak, 4), "traffic": traffic,
                     "peak_source": "measured" if peak_src == "measured" else "fallback"},
        "rows": compact_rows(kernels, next_rows, other_configs, graph),
        "gpu_launches": KERNELS_PER_STEP * args.steps,
        "clocks": clocks.summary(),
        "e2e": None if e2e is None else {k: e2e[k] for k in ("value", "unit", "h2d_bytes_per_step",
                                                             "d2h_bytes_per_step", "link_gbs", "frac_of_link")},
    }
    if not args.no_cpu_baseline and ws == 1:  # the CPU baseline runs at N = 1 only
        cb = cpu_baseline(args.cpu_sample_frac)
        cba = cpu_baseline_all_cores(args.cpu_sample_frac)
        pc = cpu_per_config(args.cpu_config_seconds)
        detail["cpu_baseline"], detail["cpu_baseline_all_cores"], detail["cpu_per_config"] = cb, cba, pc
        out["cpu_baseline"] = {k: cb[k] for k in ("value", "unit", "cores", "kind")}
        out["cpu_baseline"]["sample"] = cb["sample_short"]
        out["cpu_baseline"]["all_cores"] = {"value": cba["value"], "cores": cba["cores"]}
        out["cpu_baseline"]["per_config"] = pc["compact"]
    out["detail"] = write_detail(detail, args.detail)
    return out


def compact_rows(kernels, next_rows, other_configs, graph=None):
    """Fractions of the measured HBM peak for the other kernels, and the ring update's µs
    (from CUDA graphs like `scale_update_us` when there is a graph figure; the eager
    per-launch figure beside it).  Full figures are in the detail file."""
    r = {"multi_quantize_frac": kernels["multi_quantize_amax"]["frac_of_peak"],
         "dequantize_frac": kernels["dequantize"]["frac_of_peak"]}
    if other_configs:
        r["mlp_activation_8192x4096_frac"] = other_configs["mlp_activation"]["frac_of_peak"]
        lib = other_configs["mlp_activation"].get("same_bytes_library")
        if lib:
            r["mlp_same_bytes_copy_frac"] = lib["device_copy"]["frac_of_peak"]
        r["ragged_12_frac"] = other_configs["ragged_twelve_tensors"]["frac_of_peak"]
    if next_rows:
        r["qdq_frac"] = next_rows["qdq_amax"]["frac_of_peak"]
        r["gelu_codes_frac"] = next_rows["gelu_quantize_amax"]["codes_only"]["frac_of_peak"]
        r["layernorm_codes_frac"] = next_rows["layernorm_quantize_amax"]["codes_only"]["frac_of_peak"]
        if "layernorm_quantize_amax_wide" in next_rows:
            r["layernorm_12288_codes_frac"] = next_rows["layernorm_quantize_amax_wide"]["codes_only"]["frac_of_peak"]
        if graph:
            r["ring_update_us"] = graph["ring_update_us_after_dequantize"]
        r["ring_update_us_eager"] = next_rows["amax_scale_update_ring"]["us"]
    return r


def write_detail(detail, path):
    """Every figure of the run, as JSON, beside the printed line; returns its path."""
    p = path if os.path.isabs(path) else os.path.join(ROOT, path)
    try:
        os.makedirs(os.path.dirname(p), exist_ok=True)
        with open(p, "w") as f:
            json.dump(detail, f, indent=1)
        return os.path.relpath(p, ROOT)
    except OSError as e:
        return f"not written: {e}"


def measure_graph(args, step, stream, dev):
    """The step captured once as a CUDA graph, kernels in launch order, and replayed.

    Per-kernel events in the eager loop stop each launch from overlapping the
    previous kernel's tail, which costs a few microseconds per kernel and shows
    most on the short scale update.  Here the step runs without host launches
    or events inside; the update's own cost is taken as the difference between
    graphs of (dequantize, update) pairs and of dequantize alone.
    """
    import torch
    f = step.fp8q
    st = stream.cuda_stream

    def timed(fn, reps, replays=1):
        """us per repetition: the median over `replays` timed replays of one graph of
        `reps` repetitions (several replays of a long graph keep the event timer's
        granularity, a few us on this GPU, well below the figure's last digit)."""
        torch.cuda.synchronize(dev)  # inputs made on the default stream are complete
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(reps):
                    fn()
            for _ in range(2):
                g.replay()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(replays)]
            for e0, e1 in ev:
                e0.record(stream)
                g.replay()
                e1.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(e0.elapsed_time(e1) * 1e3 / reps for e0, e1 in ev)

    reps = max(4, min(args.steps, 50))
    step_us = timed(lambda: step.run(stream), reps)
    deq = lambda: f.fp8q_dequantize(step.grad_q, step.y_grad, f.E5M2, step.scale[4:5], st)
    upd = lambda: f.fp8q_amax_scale_update(step.hist, step.amax_new, step.scale, step.scale_inv, f.E4M3FN,
                                           f.ALGO_MAX, 0, step.slot_format, st)
    ring_hist = step.hist.clone()
    head = torch.full((S,), H - 1, dtype=torch.int32, device=dev)
    sc, si = step.scale.clone(), step.scale_inv.clone()
    ring = lambda: f.fp8q_amax_scale_update_ring(ring_hist, head, step.amax_new, sc, si, f.E4M3FN,
                                                 f.ALGO_MAX, 0, step.slot_format, st)
    tiny = torch.zeros(1, device=dev)
    deq_us = timed(deq, 100, 5)
    pair_us = timed(lambda: (deq(), upd()), 100, 5)
    ring_pair_us = timed(lambda: (deq(), ring()), 100, 5)
    # the same difference for a one-element torch fill: what any kernel node costs there
    floor_us = timed(lambda: (deq(), tiny.zero_()), 100, 5)
    return {"ms_per_step": round(step_us / 1e3, 4), "replays_of_step": reps,
            "GB/s": round(STEP_BYTES / (step_us * 1e-6) / 1e9, 1),
            "scale_update_us_after_dequantize": round(pair_us - deq_us, 3),
            "ring_update_us_after_dequantize": round(ring_pair_us - deq_us, 3),
            "one_element_fill_us_after_dequantize": round(floor_us - deq_us, 3),
            "how": "one step captured as a CUDA graph, its kernels in launch order (no branches), "
                   "CUDA events around the replay; the update's time is (dequantize+update) pairs "
                   "minus dequantize alone, both as graphs"}


def measure_other_configs(step, stream, dev, peak, warm=20, reps=50):
    """Two more quantize workloads, each launch timed on its own (mean of `reps`).

    - The MLP input activation, bf16 8192x4096 N(0,1) with 0.1% outliers x100,
      e4m3fn with the scale of the previous step's amax: its 100.7 MB of
      traffic is close to the L2 size, so a 256 MB buffer passes through L2
      before every launch and the kernel always starts from a cold L2.  Timed
      twice: after READING the buffer (L2 holds clean lines that leave for
      free) and after WRITING it (L2 full of dirty lines that the kernel's own
      traffic has to write back first, as after a producer kernel).
    - The ragged list of twelve bf16 N(0,1) tensors (2048x12288 .. 12288x4096,
      465.6 M elements) in one multi-tensor launch with the first twelve slot
      scales of the step; 1.4 GB per launch, far larger than L2.
    Algorithmic bytes: 3 per element (bf16 in, FP8 out).
    """
    import torch
    from quantize_amax_scaling_gb300 import workloads as W
    f = step.fp8q
    st = stream.cuda_stream
    out = {}

    def mean_us(launch, before=None):
        """Mean and median device time of single launches, each between its own
        events.  The event timer ticks every 2 us or so on this GPU, so a single
        launch's time is quantised; the mean over many launches (whose start is
        not tied to the tick) is not, the median is."""
        times = []
        torch.cuda.synchronize(dev)  # inputs made on the default stream are complete
        with torch.cuda.stream(stream):
            for _ in range(warm):
                if before:
                    before()
                launch()
            for _ in range(reps):
                if before:
                    before()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                launch()
                e1.record(stream)
                times.append((e0, e1))
        torch.cuda.synchronize(dev)
        us = [a.elapsed_time(b) * 1e3 for a, b in times]
        return statistics.fmean(us), statistics.median(us)

    prev = W.mlp_activation(W.SEED_MLP + 1, dev)
    sc = (prev.float().abs().max() / 448.0).reshape(1)
    del prev
    x = W.mlp_activation(W.SEED_MLP, dev).reshape(-1)
    q = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
    am = torch.zeros(1, device=dev)
    flush = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=dev)   # 256 MB, twice the L2
    nbytes = 3 * x.numel()
    launch = lambda: f.fp8q_quantize_amax(x, q, f.E4M3FN, sc, am, st)
    for key, before, how in (("mlp_activation", lambda: flush.sum(), "cold, clean: 256 MB read before every launch"),
                             ("mlp_activation_after_writes", flush.zero_,
                              "cold, dirty: 256 MB written before every launch")):
        us, us_med = mean_us(launch, before=before)
        gbs = nbytes / (us * 1e-6) / 1e9
        out[key] = {"workload": "bf16 8192x4096 N(0,1), 0.1% outliers x100 -> e4m3fn + amax",
                    "l2": how, "launches_timed": reps, "us": round(us, 3), "us_median": round(us_med, 3),
                    "GB/s": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "bytes_per_launch": nbytes}
    # Library transfers of the same 100.7 MB from the same cold, clean L2, for scale at this
    # size: torch's bf16 -> float8_e4m3fn cast of the tensor (no scale, no amax) and a
    # device-to-device copy of 50.3 MB (50.3 MB read, 50.3 MB written).
    q8 = torch.empty(x.numel(), dtype=torch.float8_e4m3fn, device=dev)
    src = torch.empty(nbytes // 2, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    lib = {}
    for key, fn in (("torch_cast_to_float8_e4m3fn", lambda: q8.copy_(x)), ("device_copy", lambda: dst.copy_(src))):
        us, us_med = mean_us(fn, before=lambda: flush.sum())
        lib[key] = {"us": round(us, 3), "us_median": round(us_med, 3),
                    "frac_of_peak": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)}
    out["mlp_activation"]["same_bytes_library"] = lib
    del x, q, flush, q8, src, dst

    xs = [t.reshape(-1) for t in W.ragged_tensors(dev)]
    qs = [torch.empty(t.numel(), dtype=torch.uint8, device=dev) for t in xs]
    ams = torch.zeros(len(xs), device=dev)
    scales = [step.scale[i:i + 1] for i in range(len(xs))]
    amaxes = [ams[i:i + 1] for i in range(len(xs))]
    us, us_med = mean_us(lambda: f.fp8q_multi_quantize_amax(xs, qs, f.E4M3FN, scales, amaxes, st))
    nbytes = 3 * sum(t.numel() for t in xs)
    gbs = nbytes / (us * 1e-6) / 1e9
    out["ragged_twelve_tensors"] = {"workload": "12 bf16 N(0,1) tensors 2048x12288 .. 12288x4096 "
                                                "(465.6 M elements) -> e4m3fn + 12 amaxes, one launch",
                                    "l2": "inputs larger than L2", "launches_timed": reps,
                                    "us": round(us, 3), "us_median": round(us_med, 3), "GB/s": round(gbs, 1),
                                    "frac_of_peak": round(gbs / peak, 4), "bytes_per_launch": nbytes}
    del xs, qs
    torch.cuda.empty_cache()
    return out


def measure_next_rows(args, step, stream, dev, peak):
    """The rows beyond the step: fp8q_qdq_amax (quantize -> dequantize in one pass), the
    GELU and LayerNorm producers, the ring update and the update fused with the next
    quantize.

    Timed with CUDA events on the launching stream over back-to-back launches, each
    launch on the next of several input/output sets (inputs larger than L2).
    """
    import torch
    f = step.fp8q
    am = torch.zeros(1, device=dev)
    n_iter = max(5, min(args.steps, 50))
    # Two buffer sets in rotation (1.6 GB for the GELU ones), so that each launch finds
    # in L2 the previous launch's dirty output, as in a stream of different kernels;
    # the same launch repeated on one buffer set overwrites those lines in L2 instead
    # (reported beside it as us_same_buffers).
    it = [0]

    def timed_loop(fn):
        torch.cuda.synchronize(dev)  # inputs made on the default stream are complete
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(n_iter):
                fn()
            s1.record(stream)
        torch.cuda.synchronize(dev)
        return s0.elapsed_time(s1) * 1e3 / n_iter

    def rot():
        it[0] = (it[0] + 1) % 2
        return it[0]

    acts = [step.act, step.act.clone()]
    ys = [torch.empty(step.act.numel(), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    us = timed_loop(lambda: f.fp8q_qdq_amax(acts[rot()], ys[it[0]], f.E4M3FN, step.scale[0:1], am,
                                            stream.cuda_stream))
    us_same = timed_loop(lambda: f.fp8q_qdq_amax(acts[0], ys[0], f.E4M3FN, step.scale[0:1], am,
                                                 stream.cuda_stream))
    nbytes = 4 * N_ACT
    gbs = nbytes / (us * 1e-6) / 1e9
    out = {"qdq_amax": {"workload": "bf16 8192x16384 -> e4m3fn -> bf16 + amax; two buffer sets in rotation",
                        "launches": n_iter, "us": round(us, 3), "GB/s": round(gbs, 1),
                        "frac_of_peak": round(gbs / peak, 4), "bytes_per_launch": nbytes,
                        "us_same_buffers": round(us_same, 3)}}
    del acts

    g = torch.Generator(device=dev)
    g.manual_seed(7)
    hs = [torch.randn(N_ACT, generator=g, device=dev).to(torch.bfloat16) for _ in range(2)]
    qs = [torch.empty(N_ACT, dtype=torch.uint8, device=dev) for _ in range(2)]
    sc0 = step.scale[0:1]
    us_q = timed_loop(lambda: f.fp8q_gelu_quantize_amax(hs[rot()], None, qs[it[0]], f.E4M3FN, sc0, am,
                                                        stream.cuda_stream))
    us_yq = timed_loop(lambda: f.fp8q_gelu_quantize_amax(hs[rot()], ys[it[0]], qs[it[0]], f.E4M3FN, sc0, am,
                                                         stream.cuda_stream))
    us_q_same = timed_loop(lambda: f.fp8q_gelu_quantize_amax(hs[0], None, qs[0], f.E4M3FN, sc0, am,
                                                             stream.cuda_stream))
    us_yq_same = timed_loop(lambda: f.fp8q_gelu_quantize_amax(hs[0], ys[0], qs[0], f.E4M3FN, sc0, am,
                                                              stream.cuda_stream))

    def unfused():
        i = rot()
        ys[i].copy_(torch.nn.functional.gelu(hs[i], approximate="tanh"))
        f.fp8q_quantize_amax(ys[i], qs[i], f.E4M3FN, sc0, am, stream.cuda_stream)
    us_unfused = timed_loop(unfused)
    out["gelu_quantize_amax"] = {
        "workload": "pre-activation bf16 8192x16384 N(0,1) -> GELU(tanh) -> e4m3fn + amax; two buffer sets in "
                    "rotation",
        "launches": n_iter,
        "codes_only": {"us": round(us_q, 3), "GB/s": round(3 * N_ACT / (us_q * 1e-6) / 1e9, 1),
                       "frac_of_peak": round(3 * N_ACT / (us_q * 1e-6) / 1e9 / peak, 4),
                       "bytes_per_launch": 3 * N_ACT, "us_same_buffers": round(us_q_same, 3)},
        "with_bf16_y": {"us": round(us_yq, 3), "GB/s": round(5 * N_ACT / (us_yq * 1e-6) / 1e9, 1),
                        "frac_of_peak": round(5 * N_ACT / (us_yq * 1e-6) / 1e9 / peak, 4),
                        "bytes_per_launch": 5 * N_ACT, "us_same_buffers": round(us_yq_same, 3)},
        "unfused_torch_gelu_then_quantize_us": round(us_unfused, 3)}
    del hs, qs, ys
    torch.cuda.empty_cache()

    # LayerNorm producer fused with the quantization on the MLP's input
    # (8192x4096): four input/output sets in rotation so that each launch reads
    # from HBM (one set is 100 MB, under the 129 MB L2), against torch's
    # layer_norm writing bf16 followed by fp8q_quantize_amax.
    from quantize_amax_scaling_gb300 import workloads as W
    rows, hid = W.SEQ * W.BATCH, W.HIDDEN
    xs = [W.residual_stream(seed=W.SEED_MLP + 7 + i, device=dev) for i in range(4)]
    qs = [torch.empty((rows, hid), dtype=torch.uint8, device=dev) for _ in range(4)]
    ys = [torch.empty((rows, hid), dtype=torch.bfloat16, device=dev) for _ in range(4)]
    gam, bet = W.layernorm_params(hid, device=dev)
    gam16, bet16 = gam.to(torch.bfloat16), bet.to(torch.bfloat16)
    it = [0]

    def ln(with_y):
        i = it[0] = (it[0] + 1) % 4
        f.fp8q_layernorm_quantize_amax(xs[i], ys[i] if with_y else None, qs[i], gam, bet, f.E4M3FN, sc0, am,
                                       stream=stream.cuda_stream)

    def ln_unfused():
        i = it[0] = (it[0] + 1) % 4
        ys[i].copy_(torch.nn.functional.layer_norm(xs[i], (hid,), gam16, bet16, eps=1e-6))
        f.fp8q_quantize_amax(ys[i], qs[i], f.E4M3FN, sc0, am, stream.cuda_stream)
    n_ln = rows * hid
    us_lq = timed_loop(lambda: ln(False))
    us_lyq = timed_loop(lambda: ln(True))
    us_lu = timed_loop(ln_unfused)
    out["layernorm_quantize_amax"] = {
        "workload": "MLP input bf16 8192x4096 -> LayerNorm (f32 gamma, beta) -> e4m3fn + amax; "
                    "4 buffer sets in rotation (400 MB, larger than L2)",
        "launches": n_iter,
        "codes_only": {"us": round(us_lq, 3), "GB/s": round(3 * n_ln / (us_lq * 1e-6) / 1e9, 1),
                       "frac_of_peak": round(3 * n_ln / (us_lq * 1e-6) / 1e9 / peak, 4),
                       "bytes_per_launch": 3 * n_ln},
        "with_bf16_y": {"us": round(us_lyq, 3), "GB/s": round(5 * n_ln / (us_lyq * 1e-6) / 1e9, 1),
                        "frac_of_peak": round(5 * n_ln / (us_lyq * 1e-6) / 1e9 / peak, 4),
                        "bytes_per_launch": 5 * n_ln},
        "unfused_torch_layer_norm_then_quantize_us": round(us_lu, 3)}
    del xs, qs, ys

    # The same producer on rows of 12288 (GPT-175B's width; thread-block clusters of 3)
    rows_w, hid_w = 2730, 12288
    xs = [W.residual_stream(seed=W.SEED_MLP + 20 + i, device=dev, shape=(rows_w, hid_w)) for i in range(4)]
    gam_w, bet_w = W.layernorm_params(hid_w, device=dev)
    qs = [torch.empty((rows_w, hid_w), dtype=torch.uint8, device=dev) for _ in range(4)]
    ys = [torch.empty((rows_w, hid_w), dtype=torch.bfloat16, device=dev) for _ in range(4)]

    def ln_w(with_y):
        i = it[0] = (it[0] + 1) % 4
        f.fp8q_layernorm_quantize_amax(xs[i], ys[i] if with_y else None, qs[i], gam_w, bet_w, f.E4M3FN, sc0, am,
                                       stream=stream.cuda_stream)
    n_w = rows_w * hid_w
    us_w, us_wy = timed_loop(lambda: ln_w(False)), timed_loop(lambda: ln_w(True))
    out["layernorm_quantize_amax_wide"] = {
        "workload": "bf16 2730x12288 (the LayerNorm input's rows) -> LayerNorm -> e4m3fn + amax, clusters of 3 "
                    "CTAs a row; 4 buffer sets in rotation",
        "codes_only": {"us": round(us_w, 3), "frac_of_peak": round(3 * n_w / (us_w * 1e-6) / 1e9 / peak, 4)},
        "with_bf16_y": {"us": round(us_wy, 3), "frac_of_peak": round(5 * n_w / (us_wy * 1e-6) / 1e9 / peak, 4)}}
    del xs, qs, ys

    # Ring-buffer update against the rolled one, each timed right after a
    # dequantize of the 8192x16384 gradient (where the update sits in the step).
    ring_hist = step.hist.clone()
    head = torch.full((S,), H - 1, dtype=torch.int32, device=dev)
    roll_hist = step.hist.clone()
    sc, si = step.scale.clone(), step.scale_inv.clone()
    times = {"ring": [], "roll": []}
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(n_iter + 3):
            for kind in ("ring", "roll"):
                f.fp8q_dequantize(step.grad_q, step.y_grad, f.E5M2, step.scale[4:5], stream.cuda_stream)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                if kind == "ring":
                    f.fp8q_amax_scale_update_ring(ring_hist, head, step.amax_new, sc, si, f.E4M3FN,
                                                  f.ALGO_MAX, 0, step.slot_format, stream.cuda_stream)
                else:
                    f.fp8q_amax_scale_update(roll_hist, step.amax_new, sc, si, f.E4M3FN, f.ALGO_MAX, 0,
                                             step.slot_format, stream.cuda_stream)
                e1.record(stream)
                if i >= 3:
                    times[kind].append((e0, e1))
    torch.cuda.synchronize(dev)
    avg = {k: sum(a.elapsed_time(b) for a, b in v) * 1e3 / len(v) for k, v in times.items()}
    ring_bytes = H * S * 4 + S * 4 * 2 + S * 4 * 4   # history read, one row + heads, scales
    out["amax_scale_update_ring"] = {
        "workload": "576 slots x history 1024, each call right after a 268 MB dequantize",
        "launches": n_iter, "us": round(avg["ring"], 3), "rolled_us_same_setting": round(avg["roll"], 3),
        "bytes_per_launch": ring_bytes}

    # The ring update fused with the next step's first quantize (the 8192x16384
    # activation with an e4m3fn slot), against the two launches it replaces:
    # back to back on the stream, and each form captured as a CUDA graph.
    slot = 6 * 40 + 1
    hs = [step.hist.clone(), step.hist.clone()]
    heads = [torch.full((S,), H - 1, dtype=torch.int32, device=dev) for _ in range(3)]
    scs = [step.scale.clone() for _ in range(2)]
    sis = [step.scale_inv.clone() for _ in range(2)]
    qf = torch.empty(N_ACT, dtype=torch.uint8, device=dev)
    amf = torch.zeros(2, device=dev)
    par = {"i": 0}

    def two_calls():
        f.fp8q_amax_scale_update_ring(hs[0], heads[0], step.amax_new, scs[0], sis[0], f.E4M3FN, f.ALGO_MAX, 0,
                                      step.slot_format, stream.cuda_stream)
        f.fp8q_quantize_amax(step.act, qf, f.E4M3FN, scs[0][slot:slot + 1], amf[0:1], stream.cuda_stream)

    def fused():
        i = par["i"] = par["i"] ^ 1
        f.fp8q_amax_scale_update_ring_quantize(hs[1], heads[1 + i], heads[2 - i], step.amax_new, scs[1], sis[1],
                                               step.act, qf, slot, amf[1:2], f.E4M3FN, f.ALGO_MAX, 0,
                                               step.slot_format, stream.cuda_stream)

    def graph_us(fn, reps=10, replays=3):
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            fn()
            stream.synchronize()
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=stream):
                for _ in range(reps):
                    fn()
            gr.replay()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(replays)]
            for e0, e1 in ev:
                e0.record(stream)
                gr.replay()
                e1.record(stream)
        torch.cuda.synchronize(dev)
        return statistics.median(e0.elapsed_time(e1) * 1e3 / reps for e0, e1 in ev)

    # The same pair on a small tensor (1024x1024), launched eagerly: the regime in
    # which one launch instead of two matters (the update's cost is launch overhead).
    xs_small = step.act[: 1 << 20]
    qs_small = torch.empty(1 << 20, dtype=torch.uint8, device=dev)

    def two_small():
        f.fp8q_amax_scale_update_ring(hs[0], heads[0], step.amax_new, scs[0], sis[0], f.E4M3FN, f.ALGO_MAX, 0,
                                      step.slot_format, stream.cuda_stream)
        f.fp8q_quantize_amax(xs_small, qs_small, f.E4M3FN, scs[0][slot:slot + 1], amf[0:1], stream.cuda_stream)

    def fused_small():
        i = par["i"] = par["i"] ^ 1
        f.fp8q_amax_scale_update_ring_quantize(hs[1], heads[1 + i], heads[2 - i], step.amax_new, scs[1], sis[1],
                                               xs_small, qs_small, slot, amf[1:2], f.E4M3FN, f.ALGO_MAX, 0,
                                               step.slot_format, stream.cuda_stream)
    out["amax_scale_update_ring_quantize_small"] = {
        "workload": "ring update of 576 slots x history 1024 + quantize of a bf16 1024x1024 tensor, launched "
                    "eagerly back to back (per call: device time between events over the loop)",
        "fused_us": round(timed_loop(fused_small), 3),
        "two_launches_us": round(timed_loop(two_small), 3),
        "fused_us_graph": round(graph_us(fused_small, 100), 3),
        "two_launches_us_graph": round(graph_us(two_small, 100), 3)}

    out["amax_scale_update_ring_quantize"] = {
        "workload": "ring update of 576 slots x history 1024 + quantize of the bf16 8192x16384 activation "
                    "with one slot's new scale",
        "launches": n_iter,
        "fused_us": round(timed_loop(fused), 3),
        "two_launches_us": round(timed_loop(two_calls), 3),
        "fused_us_graph": round(graph_us(fused), 3),
        "two_launches_us_graph": round(graph_us(two_calls), 3),
        "bytes_per_call": 3 * N_ACT + ring_bytes}
    del qf
    return out


class _HostPipeline:
    """One step from pinned host memory back to pinned host memory, in pieces.

    Each tensor is cut into pieces of CHUNK elements.  A piece is copied in on
    one stream, converted by the library call on the compute stream, and copied
    out on a third stream, so the two link directions and the kernels overlap.
    The path is elementwise and amax is max-accumulated, so the results are
    bit-identical to whole-tensor calls.  Events order every buffer's reuse
    against the previous step's use of it.
    """
    CHUNK = 64 << 20  # measured: 16M, 32M, 48M, 64M, 96M, 128M elements: 291, 296, 296.3, 298, 297.0, 297.2 GB/s

    def __init__(self, step, host_in, host_out, comp):
        import torch
        self.torch = torch
        self.s, self.hi, self.ho, self.comp = step, host_in, host_out, comp
        self.cin = torch.cuda.Stream(step.dev)
        self.cout = torch.cuda.Stream(step.dev)
        self.pieces = []
        for kind, n in (("act", step.act.numel()), ("w", step.w[0].numel()), ("grad", step.grad_q.numel())):
            for lo in range(0, n, self.CHUNK):
                self.pieces.append((kind, lo, min(n, lo + self.CHUNK)))
        assert step.w[0].numel() == step.w[1].numel()
        self.ev_k = [None] * len(self.pieces)   # previous step: kernel on the piece done
        self.ev_o = [None] * len(self.pieces)   # previous step: piece copied out
        self.ev_sc = None                       # previous step: scales copied out

    def _event(self, stream):
        e = self.torch.cuda.Event()
        e.record(stream)
        return e

    def run(self):
        torch, s, f = self.torch, self.s, self.s.fp8q
        comp, cin, cout, st = self.comp, self.cin, self.cout, self.comp.cuda_stream
        # amax_new is tiny and is read by the previous step's update: copy it on
        # the compute stream, which is already ordered after that update, so the
        # copy-in stream never waits for the end of the previous step.
        with torch.cuda.stream(comp):
            s.amax_new.copy_(self.hi["amax_new"], non_blocking=True)
            s.amax_new[:3].zero_()
        for i, (kind, lo, hi) in enumerate(self.pieces):
            with torch.cuda.stream(cin):
                if self.ev_k[i] is not None:
                    cin.wait_event(self.ev_k[i])
                if kind == "act":
                    s.act[lo:hi].copy_(self.hi["act"][lo:hi], non_blocking=True)
                elif kind == "w":
                    s.w[0][lo:hi].copy_(self.hi["w1"][lo:hi], non_blocking=True)
                    s.w[1][lo:hi].copy_(self.hi["w2"][lo:hi], non_blocking=True)
                else:
                    s.grad_q[lo:hi].copy_(self.hi["grad_q"][lo:hi], non_blocking=True)
                ev_in = self._event(cin)
            comp.wait_event(ev_in)
            if self.ev_o[i] is not None:
                comp.wait_event(self.ev_o[i])
            if kind == "act":
                f.fp8q_quantize_amax(s.act[lo:hi], s.q_act[lo:hi], f.E4M3FN, s.scale[0:1], s.amax_new[0:1], st)
            elif kind == "w":
                f.fp8q_multi_quantize_amax([s.w[0][lo:hi], s.w[1][lo:hi]], [s.q_w[0][lo:hi], s.q_w[1][lo:hi]],
                                           f.E4M3FN, [s.scale[1:2], s.scale[2:3]],
                                           [s.amax_new[1:2], s.amax_new[2:3]], st)
            else:
                f.fp8q_dequantize(s.grad_q[lo:hi], s.y_grad[lo:hi], f.E5M2, s.scale[4:5], st)
            self.ev_k[i] = self._event(comp)
            cout.wait_event(self.ev_k[i])
            with torch.cuda.stream(cout):
                if kind == "act":
                    self.ho["q_act"][lo:hi].copy_(s.q_act[lo:hi], non_blocking=True)
                elif kind == "w":
                    self.ho["q_w1"][lo:hi].copy_(s.q_w[0][lo:hi], non_blocking=True)
                    self.ho["q_w2"][lo:hi].copy_(s.q_w[1][lo:hi], non_blocking=True)
                else:
                    self.ho["y_grad"][lo:hi].copy_(s.y_grad[lo:hi], non_blocking=True)
                self.ev_o[i] = self._event(cout)
        if self.ev_sc is not None:
            comp.wait_event(self.ev_sc)
        f.fp8q_amax_scale_update(s.hist, s.amax_new, s.scale, s.scale_inv, f.E4M3FN, f.ALGO_MAX, 0,
                                 s.slot_format, st)
        cout.wait_event(self._event(comp))
        with torch.cuda.stream(cout):
            self.ho["scale"].copy_(s.scale, non_blocking=True)
            self.ho["scale_inv"].copy_(s.scale_inv, non_blocking=True)
            self.ev_sc = self._event(cout)


E2E_ROUNDS = 3


def run_e2e(args, step, stream, dev):
    """The step through the public API, from pinned host memory back to pinned host memory.

    Copies in (act, W1, W2, the FP8 gradient, amax_new) and out (the three FP8
    tensors, the dequantized gradient, scale and scale_inv) are inside the timed
    region; they overlap with the kernels in pieces (see _HostPipeline).
    """
    import torch
    steps = max(1, min(args.steps, args.e2e_steps))
    host_in = {
        "act": step.act.cpu().pin_memory(),
        "w1": step.w[0].cpu().pin_memory(),
        "w2": step.w[1].cpu().pin_memory(),
        "grad_q": step.grad_q.cpu().pin_memory(),
        "amax_new": step.amax_new.cpu().pin_memory(),
    }
    host_out = {
        "q_act": torch.empty_like(step.q_act, device="cpu").pin_memory(),
        "q_w1": torch.empty_like(step.q_w[0], device="cpu").pin_memory(),
        "q_w2": torch.empty_like(step.q_w[1], device="cpu").pin_memory(),
        "y_grad": torch.empty_like(step.y_grad, device="cpu").pin_memory(),
        "scale": torch.empty_like(step.scale, device="cpu").pin_memory(),
        "scale_inv": torch.empty_like(step.scale_inv, device="cpu").pin_memory(),
    }
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    pipe = _HostPipeline(step, host_in, host_out, stream)
    pipe.run()                                   # one untimed step
    torch.cuda.synchronize(dev)
    rounds = []
    for _ in range(E2E_ROUNDS):
        barrier()
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record(stream)
        pipe.cin.wait_event(s)
        pipe.cout.wait_event(s)
        for _ in range(steps):
            pipe.run()
        e.record(pipe.cout)          # the last copy out waits on everything before it
        torch.cuda.synchronize(dev)
        barrier()
        rounds.append(s.elapsed_time(e) / 1e3 / steps)
    ws = dist_env()[0]
    t_step = statistics.median(rounds)
    v, t = aggregate_throughput(STEP_BYTES, t_step, ws)
    link = measure_link(step, host_in, host_out, pipe, dev)
    return {"value": round(v, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": steps, "rounds": E2E_ROUNDS, "ms_per_step": round(t * 1e3, 3),
            "ms_per_step_each_round": [round(r * 1e3, 3) for r in rounds],
            "link_gbs": link["both_gbs"], "frac_of_link": round(link["both_ms"] / (t_step * 1e3), 4),
            "link": link,
            "how": f"pinned host buffers; {_HostPipeline.CHUNK >> 20}M-element pieces copied in, converted "
                   f"and copied out on three streams; {E2E_ROUNDS} timed rounds of the steps, the median "
                   "round (a host shared with other jobs can slow one); frac_of_link = time of the step's "
                   "copies alone (both directions at once, no kernels) / time of the step"}


def measure_link(step, host_in, host_out, pipe, dev, reps=3):
    """The host link alone: the step's copies (the same tensors and byte counts, whole
    tensors, pinned host memory) with no kernels, host-to-device alone, device-to-host
    alone, and both at once on two streams; the fastest of three trials of each."""
    import torch
    pairs_in = [(step.act, host_in["act"]), (step.w[0], host_in["w1"]), (step.w[1], host_in["w2"]),
                (step.grad_q, host_in["grad_q"]), (step.amax_new, host_in["amax_new"])]
    pairs_out = [(host_out["q_act"], step.q_act), (host_out["q_w1"], step.q_w[0]), (host_out["q_w2"], step.q_w[1]),
                 (host_out["y_grad"], step.y_grad), (host_out["scale"], step.scale),
                 (host_out["scale_inv"], step.scale_inv)]
    h2d = sum(h.numel() * h.element_size() for _, h in pairs_in)
    d2h = sum(h.numel() * h.element_size() for h, _ in pairs_out)

    def run(do_in, do_out):
        torch.cuda.synchronize(dev)
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        main = torch.cuda.current_stream(dev)
        s.record(main)
        pipe.cin.wait_event(s)
        pipe.cout.wait_event(s)
        for _ in range(reps):
            if do_in:
                with torch.cuda.stream(pipe.cin):
                    for d, h in pairs_in:
                        d.copy_(h, non_blocking=True)
            if do_out:
                with torch.cuda.stream(pipe.cout):
                    for h, d in pairs_out:
                        h.copy_(d, non_blocking=True)
        main.wait_stream(pipe.cin)
        main.wait_stream(pipe.cout)
        e.record(main)
        torch.cuda.synchronize(dev)
        return s.elapsed_time(e) / reps      # ms per step's copies

    run(True, True)                          # warm
    # the fastest of three trials of each: what the link can do (a host shared with
    # other jobs can slow one trial), and the smallest fraction of it for the e2e step
    trials = [(run(True, False), run(False, True), run(True, True)) for _ in range(3)]
    t_in, t_out, t_both = (min(t[i] for t in trials) for i in range(3))
    return {"h2d_gbs": round(h2d / t_in / 1e6, 1), "d2h_gbs": round(d2h / t_out / 1e6, 1),
            "both_gbs": round((h2d + d2h) / t_both / 1e6, 1), "both_ms": round(t_both, 3),
            "both_ms_each_trial": [round(t[2], 3) for t in trials],
            "h2d_bytes": h2d, "d2h_bytes": d2h}


def read_traffic():
    """DRAM bytes per launch of the quantize kernel from the committed ncu capture.

    None when there is no capture or when the code the kernel is built from
    has changed since the counters were taken (the record carries a digest of
    those sources' code).
    """
    p = os.path.join(ROOT, "profiles", "quantize_amax_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    text = ""
    for rel in d.get("sources", []):
        src = os.path.join(ROOT, rel)
        if not os.path.exists(src):
            return None
        with open(src) as f:
            text += f.read()
    if not text or source_digest(text) != d.get("source_code_sha256"):
        return None
    return d.get("dram_bytes_per_launch")


def source_digest(text: str) -> str:
    """sha256 of C/CUDA source with comments and whitespace removed (code changes only)."""
    import hashlib
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256("".join(text.split()).encode()).hexdigest()


# --------------------------------------------------------------------------- CPU oracle legs

def _oracle_sample(frac: float):
    """A bounded sample of the step for the CPU oracle: the first `frac` of each
    tensor, plus one full 576-slot update.  Returns (inputs, algorithmic bytes)."""
    import numpy as np
    import torch
    from quantize_amax_scaling_gb300 import workloads as W
    n_act = max(8, int(N_ACT * frac))
    n_w = max(8, int(N_W * frac))
    n_g = max(8, int(N_GRAD * frac))
    act = W.gelu_activation(W.SEED_FFN, "cpu", (max(1, n_act // ACT[1]) + 1, ACT[1])).reshape(-1)[:n_act]
    w = W.truncated_normal_weight((max(1, n_w // W1[1]) + 1, W1[1]), 4096, W.SEED_FFN + 10, "cpu").reshape(-1)[:n_w]
    rng = np.random.default_rng(W.SEED_GRAD)
    gq = rng.integers(0, 256, n_g, dtype=np.uint8)
    hist, new, scale, scale_inv, sf = W.scale_update_inputs("cpu")
    inputs = {"act": W.bf16_bits(act), "w": W.bf16_bits(w), "gq": gq, "hist": hist.numpy(),
              "new": new.numpy(), "scale": scale.numpy(), "scale_inv": scale_inv.numpy(), "sf": sf.numpy()}
    nbytes = BYTES_PER_ELEM * (n_act + n_w + n_g) + UPDATE_BYTES
    desc = (f"first {frac:g} of each tensor ({n_act} act + {n_w} weight elements quantized, {n_g} grad "
            f"codes dequantized) + one full 576x1024 update")
    del torch
    return inputs, nbytes, desc


def _oracle_step(inp):
    import numpy as np
    import oracle
    s = np.float32(0.0091)
    oracle.quantize_amax(inp["act"], oracle.E4M3FN, s)
    oracle.quantize_amax(inp["w"], oracle.E4M3FN, s)
    oracle.dequantize(inp["gq"], oracle.E5M2, s)
    oracle.amax_scale_update(inp["hist"], inp["new"], inp["scale"], inp["scale_inv"], oracle.E4M3FN,
                             oracle.ALGO_MAX, 0, inp["sf"])


def cpu_baseline(frac: float):
    inp, nbytes, desc = _oracle_sample(frac)
    t0 = time.perf_counter()
    _oracle_step(inp)
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": desc, "sample_short": f"first {frac:g} of each step tensor + one 576x1024 update",
            "seconds": round(dt, 3), "host": f"{os.uname().machine}, {os.cpu_count()} cores present"}


def cpu_baseline_all_cores(frac: float):
    """The same oracle sample split over every host core: each elementwise tensor in
    contiguous chunks, one thread per chunk (the oracle's C calls release the GIL;
    amax is a max, so the results are those of the whole-tensor calls), then the
    576-slot update once."""
    import numpy as np
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    inp, nbytes, desc = _oracle_sample(frac)
    n = max(1, os.cpu_count() or 1)
    s = np.float32(0.0091)

    def bounds(a, i):
        return a.size * i // n, a.size * (i + 1) // n

    def work(i):
        lo, hi = bounds(inp["act"], i)
        oracle.quantize_amax(inp["act"][lo:hi], oracle.E4M3FN, s)
        lo, hi = bounds(inp["w"], i)
        oracle.quantize_amax(inp["w"][lo:hi], oracle.E4M3FN, s)
        lo, hi = bounds(inp["gq"], i)
        oracle.dequantize(inp["gq"][lo:hi], oracle.E5M2, s)

    with ThreadPoolExecutor(n) as ex:
        t0 = time.perf_counter()
        list(ex.map(work, range(n)))
        oracle.amax_scale_update(inp["hist"], inp["new"], inp["scale"], inp["scale_inv"], oracle.E4M3FN,
                                 oracle.ALGO_MAX, 0, inp["sf"])
        dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": n, "kind": "oracle, chunks on threads",
            "sample": desc, "seconds": round(dt, 3)}


def cpu_per_config(seconds: float):
    """The oracle, as it stands, on a bounded sample of each configured workload:
    single-threaded, and split over every host core (contiguous chunks on threads;
    the oracle's C calls release the GIL; amax is a max, so the results are those of
    the whole-tensor calls).  Each sample is sized to about `seconds` of
    single-threaded work from a measured rate; GB/s counts 3 algorithmic bytes per
    element, as on the GPU.  The 576-slot update runs whole, single-threaded (its
    history is row-major over slots, so it does not split into contiguous chunks),
    for both selection algorithms and both margins."""
    import numpy as np
    import torch
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from quantize_amax_scaling_gb300 import workloads as W
    cores = max(1, os.cpu_count() or 1)
    probe = W.bf16_bits(torch.randn(1 << 20).to(torch.bfloat16))
    t0 = time.perf_counter()
    oracle.quantize_amax(probe, oracle.E4M3FN, np.float32(0.01))
    rate = probe.size / (time.perf_counter() - t0)            # elements per second, one core
    n_s = max(1 << 16, int(rate * seconds))

    def prefix(make, cols, n):
        rows = n // cols + 1
        return W.bf16_bits(make(rows, cols)).reshape(-1)[:n]

    def timed(fn, arrays):
        """(seconds on one core, seconds on all cores) of fn over every array."""
        t0 = time.perf_counter()
        for a in arrays:
            fn(a)
        t1 = time.perf_counter() - t0

        def work(i):
            for a in arrays:
                lo, hi = a.size * i // cores, a.size * (i + 1) // cores
                fn(a[lo:hi])
        with ThreadPoolExecutor(cores) as ex:
            t0 = time.perf_counter()
            list(ex.map(work, range(cores)))
            tn = time.perf_counter() - t0
        return t1, tn

    q4 = lambda a: oracle.quantize_amax(a, oracle.E4M3FN, np.float32(0.0091))
    q5 = lambda a: oracle.quantize_amax(a, oracle.E5M2, np.float32(2.0 ** -20))
    dq5 = lambda a: oracle.dequantize(a, oracle.E5M2, np.float32(2.0 ** -20))
    cases = {}
    mlp = prefix(lambda r, c: W.mlp_activation(W.SEED_MLP, "cpu", (r, c)), W.HIDDEN, n_s)
    cases["mlp_activation"] = (q4, [mlp], "bf16 8192x4096 N(0,1) with outliers -> e4m3fn + amax")
    third = n_s // 3
    ffn = [prefix(lambda r, c: W.gelu_activation(W.SEED_FFN, "cpu", (r, c)), W.FFN, third),
           prefix(lambda r, c: W.truncated_normal_weight((r, c), W.HIDDEN, W.SEED_FFN + 10, "cpu"), W.FFN, third),
           prefix(lambda r, c: W.truncated_normal_weight((r, c), W.FFN, W.SEED_FFN + 20, "cpu"), W.HIDDEN, third)]
    cases["ffn"] = (q4, ffn, "act 8192x16384 + W1 + W2 -> e4m3fn, one amax each")
    grad = prefix(lambda r, c: W.gradient((r, c), W.SEED_GRAD, "cpu"), W.FFN, n_s)
    cases["grad_quantize"] = (q5, [grad], "gradients sign x lognormal(-12, 3) -> e5m2 saturating")
    gq, _ = oracle.quantize_amax(grad, oracle.E5M2, np.float32(2.0 ** -20))
    cases["grad_dequantize"] = (dq5, [gq], "e5m2 codes -> bf16")
    per = max(1, n_s // 12)
    rag = [W.bf16_bits(t).reshape(-1)[:per] for t in W.ragged_tensors("cpu", scale_down=max(1, (2048 * 12288) // per))]
    cases["ragged_12"] = (q4, rag, "12 ragged bf16 tensors -> e4m3fn, one amax each")
    out, compact = {}, {"cores": cores}
    for name, (fn, arrays, what) in cases.items():
        n = sum(a.size for a in arrays)
        t1, tn = timed(fn, arrays)
        g1, gn = 3 * n / t1 / 1e9, 3 * n / tn / 1e9
        out[name] = {"workload": what, "elements_sampled": int(n), "GB/s_1_core": round(g1, 4),
                     f"GB/s_{cores}_cores": round(gn, 4), "seconds_1_core": round(t1, 3)}
        compact[name] = [round(g1, 4), round(gn, 4)]
    hist, new, sc, si, sf = W.scale_update_inputs("cpu")
    ups = {}
    for algo in (oracle.ALGO_MAX, oracle.ALGO_MOST_RECENT):
        for margin in (0, 1):
            h, a, b = hist.numpy().copy(), sc.numpy().copy(), si.numpy().copy()
            t0 = time.perf_counter()
            oracle.amax_scale_update(h, new.numpy(), a, b, oracle.E4M3FN, algo, margin, sf.numpy())
            ups[f"{'max' if algo == 0 else 'most_recent'}_m{margin}"] = round((time.perf_counter() - t0) * 1e6, 1)
    out["update_576x1024_us_1_core"] = ups
    compact["update_us"] = list(ups.values())
    return {"configs": out, "compact": compact, "sample_seconds": seconds,
            "host": f"{os.uname().machine}, {cores} cores, {cpu_model()}"}


def cpu_model() -> str:
    """The host CPU's model name, as lscpu or /proc/cpuinfo give it ("" if neither)."""
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return ""


def run_reference(args):
    """The CPU oracle, as it stands, timed on the host on a bounded sample per step."""
    inp, nbytes, desc = _oracle_sample(args.ref_sample_frac)
    for _ in range(args.warmup):
        _oracle_step(inp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(inp)
    dt = (time.perf_counter() - t0) / args.steps
    v = nbytes / dt / 1e9
    return {"metric": METRIC, "impl": "reference", "value": round(v, 4), "unit": "GB/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded)", "config": {"workload": WORKLOAD, "step_bytes_sampled": nbytes},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


CASES = ("quantize_8192x16384", "quantize_8192x4096", "dequantize_8192x16384", "update_576x1024",
         "gelu_8192x16384", "gelu_y_8192x16384", "layernorm_8192x4096", "layernorm_4096x8192",
         "qdq_8192x16384")


def run_case(name: str, launches: int):
    """One kernel on its benchmark workload, `launches` times back to back, then exit:
    the program a profiler captures (ncu -k <kernel> -s 1 -c 1 ...).  The 100 MB
    quantize case reads 256 MB before each launch, so that it starts from a cold L2,
    as in the bench's other_configs."""
    import torch
    from quantize_amax_scaling_gb300 import fp8q as f
    from quantize_amax_scaling_gb300 import workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sc = torch.full((1,), 0.0091, device=dev)
    am = torch.zeros(1, device=dev)
    before = None
    if name == "quantize_8192x16384":
        x = W.gelu_activation(W.SEED_FFN, dev).reshape(-1)
        q = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
        launch = lambda: f.fp8q_quantize_amax(x, q, f.E4M3FN, sc, am)
    elif name == "quantize_8192x4096":
        x = W.mlp_activation(W.SEED_MLP, dev).reshape(-1)
        q = torch.empty(x.numel(), dtype=torch.uint8, device=dev)
        flush = torch.zeros(64 * 1024 * 1024, dtype=torch.int32, device=dev)
        before = lambda: flush.sum()
        launch = lambda: f.fp8q_quantize_amax(x, q, f.E4M3FN, sc, am)
    elif name == "dequantize_8192x16384":
        g = W.gradient(GRAD, W.SEED_GRAD, dev).reshape(-1)
        q = torch.empty(g.numel(), dtype=torch.uint8, device=dev)
        f.fp8q_quantize_amax(g, q, f.E5M2, sc, am)
        y = torch.empty(g.numel(), dtype=torch.bfloat16, device=dev)
        launch = lambda: f.fp8q_dequantize(q, y, f.E5M2, sc)
    elif name == "update_576x1024":
        hist, new, scale, scale_inv, sf = W.scale_update_inputs(dev)
        launch = lambda: f.fp8q_amax_scale_update(hist, new, scale, scale_inv, f.E4M3FN, f.ALGO_MAX, 0, sf)
    elif name in ("gelu_8192x16384", "gelu_y_8192x16384"):
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        h = torch.randn(N_ACT, generator=g, device=dev).to(torch.bfloat16)
        q = torch.empty(N_ACT, dtype=torch.uint8, device=dev)
        y = torch.empty(N_ACT, dtype=torch.bfloat16, device=dev) if name == "gelu_y_8192x16384" else None
        launch = lambda: f.fp8q_gelu_quantize_amax(h, y, q, f.E4M3FN, sc, am)
    elif name in ("layernorm_8192x4096", "layernorm_4096x8192"):
        x = W.residual_stream(device=dev, shape=(8192, 4096) if name == "layernorm_8192x4096" else (4096, 8192))
        gam, bet = W.layernorm_params(x.shape[1], device=dev)
        q = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        launch = lambda: f.fp8q_layernorm_quantize_amax(x, None, q, gam, bet, f.E4M3FN, sc, am)
    elif name == "qdq_8192x16384":
        x = W.gelu_activation(W.SEED_FFN, dev).reshape(-1)
        y = torch.empty(x.numel(), dtype=torch.bfloat16, device=dev)
        launch = lambda: f.fp8q_qdq_amax(x, y, f.E4M3FN, sc, am)
    else:
        raise ValueError(name)
    for _ in range(launches):
        if before:
            before()
        launch()
    torch.cuda.synchronize(dev)
    return {"case": name, "launches": launches, "amax": float(am)}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["fp8q", "reference"], default="fp8q")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the CUDA-graph and next-row measurements (run after the timed region)")
    ap.add_argument("--cpu-sample-frac", type=float, default=0.4)  # about 10 s of oracle work
    ap.add_argument("--ref-sample-frac", type=float, default=1.0 / 128)
    ap.add_argument("--case", choices=CASES, default=None,
                    help="launch one kernel on its benchmark workload --launches times and exit (for profilers)")
    ap.add_argument("--launches", type=int, default=2)
    ap.add_argument("--detail", default="bench_detail.json",
                    help="where every figure of the run is written as JSON (the printed line is the summary)")
    ap.add_argument("--cpu-config-seconds", type=float, default=1.0,
                    help="about this much single-core oracle work per config of the per-config CPU baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    ws, rank, local = dist_env()
    if args.case:
        print(json.dumps(run_case(args.case, args.launches)), flush=True)
        return 0
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    out = run_gpu(args, ws, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
