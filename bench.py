"""Benchmark of the block-quantized GEMV on GB300.

Default workload (the headline): one decode step through a 32-layer
Q4_K_M-style stack -- per layer Q4_K q/k/v/o 4096 x 4096, Q4_K gate/up
11008 x 4096, Q6_K down 4096 x 11008 -- each matrix with its own fresh
activation vector (n_vec = 1; no chaining between matrices). A step is the
224 matrix-vector products with their activation quantization to Q8_K. The
products are independent, so the step runs them as batched calls
(qgemv_batched: one launch for the 192 Q4_K matrices of row length 4096,
one for the 32 Q6_K matrices of row length 11008); the same step with one
qgemv call per matrix is reported beside it ("per_call"). Weights stay
resident in HBM (4.01 GB, far above L2, so every step streams them from HBM).
The metric is effective weight bandwidth: weight bytes streamed per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--n-vec V]

Prints one JSON line (rank 0). Under torchrun every rank runs the whole
workload on its own GPU (replicas: weak scaling); value sums all ranks' bytes
over the slowest rank's time.
"""
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

METRIC = "Q4_K/Q6_K GEMV effective weight GB/s (% of GB300 HBM peak)"
UNIT = "GB/s"


# ----------------------------------------------------------------- helpers
# Replicas under torchrun: each rank runs the whole workload on its own GPU;
# the timed regions start together and the job's time is its slowest rank's.
def rank_barrier(world):
    """All ranks meet here (nothing to do with one process)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(t, world, device="cpu"):
    """The slowest rank's time, returned on every rank."""
    if world <= 1:
        return t
    import torch
    import torch.distributed as dist
    tt = torch.tensor([t], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_rate(units_per_step, steps, world, seconds, scale=1e9):
    """Units that all ranks processed per second, over the slowest rank's
    time (every rank processes units_per_step per step)."""
    return units_per_step * steps * world / seconds / scale


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_family(kernel_desc):
    """'tc' for the tcgen05 kernel, 'mma' for the mma.sync tensor-core kernel,
    'dp4a' for the streaming __dp4a one."""
    if kernel_desc.startswith("gemv_tc"):
        return "tc"
    return "mma" if kernel_desc.startswith("gemv_mma") else "dp4a"


def kernel_source_hash(family):
    """Hash of the sources of one GEMV kernel family (to tell whether a
    committed ncu traffic figure still describes the current kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ggml_block_quantized_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if family == "gemm":  # the prefill GEMMs
            mine = name.startswith("gemm") or name == "tc_common.cuh"
        elif family in ("mma", "tc"):
            mine = name.startswith("gemv_" + family)
        else:
            mine = name.startswith("gemv") and not name.startswith(("gemv_mma", "gemv_tc"))
        if mine or name == "qg_common.cuh":
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def committed_traffic(kernel_key, family):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current sources of the kernel's family; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(kernel_key)
        if e and e.get("source_hash") == kernel_source_hash(family):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ the workload
def build_workload(name, n_vec, device, keep_host_layers=2, n_layers=None):
    """Device-resident inputs for every qgemv call of one step.

    Returns (calls, host_sample): calls is a list of dicts (type, n_out, n_in,
    W, x, y) on the device; host_sample keeps the host arrays of the first
    calls for the CPU baseline."""
    import torch

    import ggml_block_quantized_gb300 as qg
    from ggml_block_quantized_gb300 import synth

    calls, host_sample = [], []
    if name == "layer_stack":
        for layer in range(synth.N_LAYERS if n_layers is None else n_layers):
            for m in range(len(synth.LAYER_MATRICES)):
                mat = synth.layer_matrix(layer, m, n_vec)
                c = dict(kind=mat["name"], type=mat["type"], n_out=mat["n_out"], n_in=mat["n_in"],
                         W=torch.from_numpy(mat["w_blocks"]).to(device),
                         x=torch.from_numpy(mat["x"]).to(device))
                calls.append(c)
                if layer < keep_host_layers:
                    host_sample.append(dict(type=mat["type"], n_out=mat["n_out"], n_in=mat["n_in"],
                                            W=mat["w_blocks"], x=mat["x"]))
    else:
        m = synth.single_matrix(name, n_vec=n_vec)
        t = m["type"]
        if "w_f32" in m:
            W = qg.quantize_rows(t, torch.from_numpy(m["w_f32"]).to(device), m["n_out"])
        else:
            W = torch.from_numpy(m["w_blocks"]).to(device)
        torch.cuda.synchronize()
        # enough distinct copies of the weights that the rotation exceeds 4x L2
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        copies = max(1, int(np.ceil(4 * l2 / W.numel())))
        x = torch.from_numpy(m["x"]).to(device)
        for i in range(copies):
            calls.append(dict(kind=name, type=t, n_out=m["n_out"], n_in=m["n_in"],
                              W=W if i == 0 else W.clone(), x=x))
        host_sample.append(dict(type=t, n_out=m["n_out"], n_in=m["n_in"], W=W.cpu().numpy(), x=m["x"]))
    # every x and every y of the step in one contiguous buffer each (views per
    # matrix), laid out group by group (type, row length: the batched
    # launches) so that each launch's inputs and outputs are one range
    xs_len = sum(c["x"].numel() for c in calls)
    ys_len = sum(n_vec * c["n_out"] for c in calls)
    X = torch.empty(xs_len, dtype=torch.float32, device=device)
    Y = torch.empty(ys_len, dtype=torch.float32, device=device)
    xo = yo = 0
    for c in sorted(calls, key=lambda c: (c["type"], c["n_in"])):  # stable: call order within a group
        n = c["x"].numel()
        X[xo:xo + n].copy_(c["x"])
        c["x"] = X[xo:xo + n]
        c["y"] = Y[yo:yo + n_vec * c["n_out"]].view(n_vec, c["n_out"])
        c["x_off"], c["y_off"] = xo, yo
        xo += n
        yo += n_vec * c["n_out"]
    torch.cuda.synchronize()
    return calls, host_sample, X, Y


def weight_bytes(calls):
    return sum(c["W"].numel() for c in calls)


# ------------------------------------------------------------ CPU baseline
def time_oracle(sample, n_vec, budget_s=12.0):
    """The oracle as it stands, rows split over the host cores; returns
    (GB/s of weight bytes, cores, description)."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    cores = len(os.sched_getaffinity(0))
    done_bytes, t_total, ncalls = 0, 0.0, 0
    with ThreadPoolExecutor(max_workers=cores) as ex:
        for c in sample:
            t0 = time.perf_counter()
            at = oracle.act_type(c["type"])
            xq = oracle.quantize(at, c["x"])
            y = np.zeros((n_vec, c["n_out"]))
            chunks = np.linspace(0, c["n_out"], cores * 4 + 1).astype(int)
            list(ex.map(lambda r: oracle.gemv(c["type"], c["W"], xq, c["n_out"], c["n_in"], n_vec,
                                              rows=(int(r[0]), int(r[1])), out=y),
                        zip(chunks[:-1], chunks[1:])))
            t_total += time.perf_counter() - t0
            done_bytes += c["W"].size
            ncalls += 1
            if t_total > budget_s:
                break
    return done_bytes / t_total / 1e9, cores, f"{ncalls} of the step's qgemv calls (first layers), n_vec={n_vec}"


# ------------------------------------------------- every workload, one line
SINGLE_CONFIGS = ["q8_0_256x1024", "q4_0_4096", "q4_k_4096", "q6_k_32000"]   # the four single-matrix workloads
L2_HOT = ("q8_0_256x1024", "q4_0_4096", "q4_k_4096")  # small enough to also time with W resident in L2
OTHER_TYPES = ["q4_1_32000", "q5_0_32000", "q2_k_32000", "q3_k_32000", "q5_k_32000"]


def time_single_calls(qg, timer, t, n_out, n_in, nv, W, x, peak, reps=10, l2_hot=False):
    """One qgemv call per weight copy, the copies rotating through more than
    4x L2 so every call streams W from HBM; returns the per-call figures.
    With l2_hot the same number of calls all use W itself, which stays in L2
    after the first call (a latency figure, not a bandwidth one)."""
    import torch
    dev = W.device
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    copies = max(1, int(np.ceil(4 * l2 / W.numel())))
    Ws = [W] * copies if l2_hot else [W] + [W.clone() for _ in range(copies - 1)]
    y = torch.empty((nv, n_out), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, qg.qgemv_workspace_bytes(t, n_in, nv)), dtype=torch.uint8, device=dev)

    def fn():
        for Wc in Ws:
            qg.qgemv(t, Wc, x, n_out, n_in, nv, y=y, workspace=ws, stream=timer.stream)
    g = timer.capture(fn)
    tt, _ = timer.time(g, reps)
    del g, Ws
    per = tt / (reps * copies)
    gbs = W.numel() / per / 1e9
    info = qg.kernel_info(t, n_out, n_in, nv, 1)
    return {"us_per_call": round(per * 1e6, 3), "GB_s": round(gbs, 1), "frac": round(gbs / peak, 4),
            "launches_per_call": 1 if "fused-quantize" in info else 2, "kernel": info,
            "weight_bytes": int(W.numel()), "copies_rotated": copies}


def measure_single_workloads(qg, synth, timer, device, peak, names):
    """Each single-matrix workload at one and eight vectors (same weights)."""
    import torch
    out = {}
    for name in names:
        m = synth.single_matrix(name, n_vec=8)
        t, n_out, n_in = m["type"], m["n_out"], m["n_in"]
        if "w_f32" in m:
            W = qg.quantize_rows(t, torch.from_numpy(m["w_f32"]).to(device), n_out, stream=timer.stream)
        else:
            W = torch.from_numpy(m["w_blocks"]).to(device)
        x8 = torch.from_numpy(m["x"]).to(device)
        torch.cuda.synchronize()
        row = {"shape": f"{qg.TYPE_NAMES[t]} {n_out}x{n_in}"}
        for nv in (1, 8):
            row[f"n_vec={nv}"] = time_single_calls(qg, timer, t, n_out, n_in, nv, W, x8[:nv * n_in], peak)
            if name in L2_HOT:
                hot = time_single_calls(qg, timer, t, n_out, n_in, nv, W, x8[:nv * n_in], peak, l2_hot=True)
                row[f"n_vec={nv}"]["l2_hot"] = {"us_per_call": hot["us_per_call"],
                                                "note": "one weight copy, resident in L2 after the first call"}
        if name == "q4_k_4096":
            row["dequantize_rows"] = time_dequantize(qg, timer, t, n_out, n_in, W, peak)
        out[name] = row
        del W, x8, m
        torch.cuda.synchronize()
    return out


def time_dequantize(qg, timer, t, n_out, n_in, W, peak, reps=10):
    """dequantize_rows, read + write bytes over the time; weight copies and
    outputs rotate through buffers larger than L2."""
    import torch
    dev = W.device
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    n_el = n_out * n_in
    n_outs = max(2, int(np.ceil(2 * l2 / (4 * n_el))))
    outs = [torch.empty((n_out, n_in), dtype=torch.float32, device=dev) for _ in range(n_outs)]
    Ws = [W] + [W.clone() for _ in range(max(1, int(np.ceil(2 * l2 / W.numel()))) - 1)]
    seq = [(Ws[i % len(Ws)], outs[i % n_outs]) for i in range(max(len(Ws), n_outs))]

    def fn():
        for w, o in seq:
            qg.dequantize_rows(t, w, n_out, n_in, out=o, stream=timer.stream)
    g = timer.capture(fn)
    td, _ = timer.time(g, reps)
    del g, outs, Ws
    per = td / (reps * len(seq))
    moved = W.numel() + 4 * n_el
    return {"us_per_call": round(per * 1e6, 3), "bytes_per_call": int(moved), "GB_s": round(moved / per / 1e9, 1),
            "frac": round(moved / per / 1e9 / peak, 4),
            "note": "read + write bytes over the time; weights and outputs rotate through buffers larger than L2"}


def layer_groups(calls):
    """One decoder layer's launches in dependency order: q/k/v batched, o,
    gate/up batched, down (calls are in layer order, 7 per layer)."""
    out = []
    for base in range(0, len(calls), 7):
        lc = calls[base:base + 7]
        out += [lc[0:3], lc[3:4], lc[4:6], lc[6:7]]
    return out


def time_decode_chain(qg, timer, calls, nv, wbytes, peak, reps):
    """The stack as a decoder runs it: every launch waits for the one before
    it on the stream (q/k/v batched, o, gate/up batched, down per layer)."""
    import torch
    dev = calls[0]["W"].device
    ws = torch.empty(max(qg.qgemv_workspace_bytes(c["type"], c["n_in"], nv) for c in calls) * 3,
                     dtype=torch.uint8, device=dev)
    steps, launches = [], 0
    for grp in layer_groups(calls):
        c0 = grp[0]
        if len(grp) == 1:
            steps.append(("one", c0))
        else:
            steps.append(("batch", qg.BatchPlan(c0["type"], [(c["W"], c["x"], c["y"], c["n_out"]) for c in grp],
                                                c0["n_in"], nv, workspace=ws)))
        info = qg.kernel_info(c0["type"], sum(c["n_out"] for c in grp), c0["n_in"], nv, len(grp))
        launches += 1 if "fused-quantize" in info else 2

    def fn():
        for kind, v in steps:
            if kind == "one":
                qg.qgemv(v["type"], v["W"], v["x"], v["n_out"], v["n_in"], nv, y=v["y"], workspace=ws,
                         stream=timer.stream)
            else:
                v.run(timer.stream)
    g = timer.capture(fn)
    tt, _ = timer.time(g, reps)
    del g
    gbs = wbytes * reps / tt / 1e9
    return {"value": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / peak, 4),
            "ms_per_step": round(tt / reps * 1e3, 4), "launches_per_step": launches,
            "api": "per layer: qgemv_batched(q, k, v), qgemv(o), qgemv_batched(gate, up), qgemv(down); "
                   "stream-ordered, each launch after the previous one"}


class GraphTimer:
    """CUDA-graph capture and CUDA-event timing on one stream."""

    def __init__(self, stream, world, device):
        self.stream, self.world, self.device = stream, world, device

    def capture(self, fn):
        import torch
        with torch.cuda.stream(self.stream):
            fn()  # eager warm-up on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            fn()
        return g

    def time(self, g, reps, sampler=None):
        import torch
        with torch.cuda.stream(self.stream):
            for _ in range(2):
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if sampler:
            sampler.start()
        rank_barrier(self.world)
        torch.cuda.synchronize()
        with torch.cuda.stream(self.stream):
            e0.record(self.stream)
            for _ in range(reps):
                g.replay()
            e1.record(self.stream)
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        return max_over_ranks(e0.elapsed_time(e1) / 1e3, self.world, self.device), clocks


# --------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch

    import __graft_entry__
    import ggml_block_quantized_gb300 as qg

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    calls, host_sample, X, Y = build_workload(args.workload, args.n_vec, device, n_layers=args.layers)
    wbytes = weight_bytes(calls)
    nv = args.n_vec
    ws = torch.empty(max(qg.qgemv_workspace_bytes(c["type"], c["n_in"], nv) for c in calls),
                     dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)

    # Batched plans: matrices grouped by (type, n_in), at most MAX_BATCH a launch.
    groups = {}
    for c in calls:
        groups.setdefault((c["type"], c["n_in"]), []).append(c)
    plans = []
    for (t, n_in), cs in sorted(groups.items()):
        for i in range(0, len(cs), qg.MAX_BATCH):
            part = cs[i:i + qg.MAX_BATCH]
            plans.append((t, part, qg.BatchPlan(t, [(c["W"], c["x"], c["y"], c["n_out"]) for c in part], n_in, nv)))
    batched = args.workload == "layer_stack"

    def step_batched():
        for _, _, plan in plans:
            plan.run(stream)

    def step_calls(sel=None):
        for c in (calls if sel is None else sel):
            qg.qgemv(c["type"], c["W"], c["x"], c["n_out"], c["n_in"], nv, y=c["y"], workspace=ws, stream=stream)

    timer = GraphTimer(stream, 1, device)  # per-rank times; the headline takes the max over ranks below
    capture, time_graph = timer.capture, timer.time

    step = step_batched if batched else step_calls
    g_step = capture(step)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g_step.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    t, clocks = time_graph(g_step, args.steps, sampler)
    t = max_over_ranks(t, world, device)
    value = whole_job_rate(wbytes, args.steps, world, t)
    ms_per_step = t / args.steps * 1e3
    assert qg.device_error() == 0, "a kernel reported a bounded-wait timeout"
    # a product whose plan quantizes x in its prologue is one launch, else two
    def launches_of(t, rows, n_in, n_mats):
        return 1 if "fused-quantize" in qg.kernel_info(t, rows, n_in, nv, n_mats) else 2
    if batched:
        launches_per_step = sum(launches_of(t, sum(c["n_out"] for c in part), part[0]["n_in"], len(part))
                                for t, part, _ in plans)
    else:
        launches_per_step = sum(launches_of(c["type"], c["n_out"], c["n_in"], 1) for c in calls)
    del g_step

    # ---- one qgemv call per matrix (stream-ordered, each call may depend on the previous)
    per_call = None
    if batched:
        g = capture(step_calls)
        reps = max(3, args.steps // 4)
        tc, _ = time_graph(g, reps)
        del g
        per_call = {"value": round(wbytes * reps / tc / 1e9, 1), "unit": UNIT,
                    "ms_per_step": round(tc / reps * 1e3, 4),
                    "launches_per_step": sum(launches_of(c["type"], c["n_out"], c["n_in"], 1) for c in calls)}

    # ---- dequantize_rows on the same weights (the Q4_K 4096 x 4096
    # workload's second operation): read W, write every element as f32;
    # the outputs rotate through buffers larger than L2 together
    dequant = None
    if args.workload == "q4_k_4096":
        c0 = calls[0]
        n_el = c0["n_out"] * c0["n_in"]
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n_outs = max(2, int(np.ceil(2 * l2 / (4 * n_el))))
        outs = [torch.empty((c0["n_out"], c0["n_in"]), dtype=torch.float32, device=device) for _ in range(n_outs)]
        seq = [(c["W"], outs[i % n_outs]) for i, c in enumerate(calls)]

        def deq_step():
            for w, o in seq:
                qg.dequantize_rows(c0["type"], w, c0["n_out"], c0["n_in"], out=o, stream=stream)
        g = capture(deq_step)
        reps = max(3, args.steps // 4)
        td, _ = time_graph(g, reps)
        td = max_over_ranks(td, world, device)
        del g, outs
        per = td / (reps * len(seq))
        moved = c0["W"].numel() + 4 * n_el
        dequant = {"us_per_call": round(per * 1e6, 3), "bytes_per_call": int(moved),
                   "GB_s": round(moved / per / 1e9, 1), "hbm_frac": round(moved / per / 1e9 / measured_peaks()[0], 4),
                   "note": "read + write bytes over the time; outputs rotate through buffers larger than L2"}

    # ---- per-kind breakdown: each kind's calls alone, one qgemv call each
    peak, peak_kind = measured_peaks()
    breakdown = {}
    kinds = sorted({(c["kind"] if c["kind"] not in ("q", "k", "v", "o") else "qkvo") for c in calls})
    for kind in kinds:
        sel = [c for c in calls if (c["kind"] == kind or (kind == "qkvo" and c["kind"] in ("q", "k", "v", "o")))]
        g = capture(lambda sel=sel: step_calls(sel))
        reps = max(3, min(50, int(0.3 / max(1e-6, ms_per_step / 1e3 * len(sel) / len(calls)))))
        tk, _ = time_graph(g, reps)
        b = weight_bytes(sel)
        c0 = sel[0]
        breakdown[kind] = {"shape": f"{qg.TYPE_NAMES[c0['type']]} {c0['n_out']}x{c0['n_in']}",
                           "calls_per_step": len(sel), "us_per_call": round(tk / reps / len(sel) * 1e6, 3),
                           "GB_s": round(b * reps / tk / 1e9, 1), "frac": round(b * reps / tk / 1e9 / peak, 4),
                           "kernel": qg.kernel_info(c0["type"], c0["n_out"], c0["n_in"], nv, 1)}
        del g

    # ---- roofline of the dominant kernel: the launch that streams the most
    # weight bytes, timed alone; algorithmic bytes = its weights + f32
    # activations read + f32 outputs written
    peak, peak_kind = measured_peaks()
    if batched:
        dom_t, dom_calls, dom_plan = max(plans, key=lambda pl: weight_bytes(pl[1]))
        g = capture(lambda: dom_plan.run(stream))
        launches = 1
    else:
        dom_t = calls[0]["type"]
        dom_calls = calls
        g = capture(step_calls)
        launches = len(calls)
    reps = 10
    tg, _ = time_graph(g, reps)
    del g
    alg_bytes = sum(c["W"].numel() + 4 * nv * (c["n_in"] + c["n_out"]) for c in dom_calls)
    per_launch = alg_bytes / launches
    avg_dur = tg / reps / launches
    achieved = per_launch / avg_dur / 1e9
    rows = sum(c["n_out"] for c in dom_calls) if batched else dom_calls[0]["n_out"]
    desc = qg.kernel_info(dom_t, rows, dom_calls[0]["n_in"], nv, len(dom_calls) if batched else 1)
    kernel_key = desc.split(" ")[0]
    roofline = {"bound": "hbm", "kernel": desc + (" (batched launch)" if batched else ""),
                "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": committed_traffic(f"{kernel_key}@{args.workload}", kernel_family(desc)),
                "algorithmic_bytes_per_launch": int(per_launch), "avg_launch_us": round(avg_dur * 1e6, 3),
                "launches": launches}

    # ---- every workload of the benchmark in the same line: the four
    # single-matrix workloads and the other weight types at one and eight
    # vectors, dequantize_rows, the stack at eight vectors, and the stack as
    # a decoder runs it (dependency-ordered launches)
    configs = None
    if batched and args.configs:
        import torch as _t
        from ggml_block_quantized_gb300 import synth
        t_cfg = time.perf_counter()
        configs = {}
        chain_reps = max(3, args.steps // 4)
        configs["decode_chain"] = {f"n_vec={nv}": time_decode_chain(qg, timer, calls, nv, wbytes, peak, chain_reps)}
        if nv == 1 and args.layers in (None, synth.N_LAYERS):
            nv8 = 8
            xs8 = [synth.layer_x(layer, m, nv8) for layer in range(synth.N_LAYERS)
                   for m in range(len(synth.LAYER_MATRICES))]
            X8 = _t.from_numpy(np.concatenate(xs8)).to(device)
            Y8 = _t.empty(sum(nv8 * c["n_out"] for c in calls), dtype=_t.float32, device=device)
            calls8, xo, yo = [], 0, 0
            for c, xh in zip(calls, xs8):
                c8 = dict(c)
                c8["x"] = X8[xo:xo + xh.size]
                c8["y"] = Y8[yo:yo + nv8 * c["n_out"]].view(nv8, c["n_out"])
                xo += xh.size
                yo += nv8 * c["n_out"]
                calls8.append(c8)
            del xs8
            groups8 = {}
            for c in calls8:
                groups8.setdefault((c["type"], c["n_in"]), []).append(c)
            plans8 = []
            for (ty8, n_in8), cs in sorted(groups8.items()):
                for i in range(0, len(cs), qg.MAX_BATCH):
                    part = cs[i:i + qg.MAX_BATCH]
                    plans8.append((ty8, part, qg.BatchPlan(ty8, [(c["W"], c["x"], c["y"], c["n_out"]) for c in part],
                                                           n_in8, nv8)))
            g = capture(lambda: [pl.run(stream) for _, _, pl in plans8])
            t8, _ = time_graph(g, chain_reps)
            del g
            d_t, d_calls, d_plan = max(plans8, key=lambda pl: weight_bytes(pl[1]))
            g = capture(lambda: d_plan.run(stream))
            tg8, _ = time_graph(g, 10)
            del g
            alg8 = sum(c["W"].numel() + 4 * nv8 * (c["n_in"] + c["n_out"]) for c in d_calls)
            desc8 = qg.kernel_info(d_t, sum(c["n_out"] for c in d_calls), d_calls[0]["n_in"], nv8, len(d_calls))
            v8 = wbytes * chain_reps / t8 / 1e9
            configs["layer_stack_n_vec=8"] = {
                "value": round(v8, 1), "unit": UNIT, "frac": round(v8 / peak, 4),
                "ms_per_step": round(t8 / chain_reps * 1e3, 4),
                "api": "qgemv_batched (one launch per type and row length)",
                "roofline": {"bound": "hbm", "kernel": desc8 + " (batched launch)",
                             "achieved": round(alg8 / (tg8 / 10) / 1e9, 1), "peak": peak, "unit": "GB/s",
                             "frac": round(alg8 / (tg8 / 10) / 1e9 / peak, 4),
                             "traffic": committed_traffic(f"{desc8.split(' ')[0]}@layer_stack_nv8",
                                                          kernel_family(desc8)),
                             "algorithmic_bytes_per_launch": int(alg8), "avg_launch_us": round(tg8 / 10 * 1e6, 3)}}
            configs["decode_chain"]["n_vec=8"] = time_decode_chain(qg, timer, calls8, nv8, wbytes, peak, chain_reps)
            del plans8, calls8, groups8, X8, Y8
            _t.cuda.synchronize()
        configs.update(measure_single_workloads(qg, synth, timer, device, peak, SINGLE_CONFIGS + OTHER_TYPES))
        configs["seconds"] = round(time.perf_counter() - t_cfg, 1)

    # ---- end to end through the public API with host buffers: each step
    # copies all of its x in from pinned host memory (one copy) and all of
    # its y back out (one copy)
    HX = X.cpu().pin_memory()
    HY = torch.empty(Y.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        X.copy_(HX, non_blocking=True)
        step()
        HY.copy_(Y, non_blocking=True)

    if batched:
        # The launches' inputs come in and their outputs go out on a copy
        # stream, each launch waiting only for its own inputs: the copies of
        # the later group overlap the earlier group's compute (every byte
        # still crosses between host and device each step).
        copy_stream = torch.cuda.Stream(device)
        # with several vectors the copies are large: launches of at most 48
        # matrices, so that the inputs exposed before the first launch and
        # the outputs after the last are small (with one vector a smaller
        # launch costs more than the copy it hides)
        per_launch = 48 if nv > 2 else qg.MAX_BATCH
        # the step's first launch may be shorter (--e2e-head matrices), so that
        # the compute starts after a small part of the inputs has arrived
        e2e_plans = []
        for gi, ((t, n_in), cs) in enumerate(sorted(groups.items())):
            i = 0
            while i < len(cs):
                n = args.e2e_head if gi == 0 and i == 0 and args.e2e_head > 0 else per_launch
                part = cs[i:i + n]
                i += n
                e2e_plans.append((t, part, qg.BatchPlan(t, [(c["W"], c["x"], c["y"], c["n_out"]) for c in part],
                                                        n_in, nv)))
        spans = []
        for _, part, _ in e2e_plans:
            x0 = min(c["x_off"] for c in part)
            x1 = max(c["x_off"] + c["x"].numel() for c in part)
            y0 = min(c["y_off"] for c in part)
            y1 = max(c["y_off"] + c["y"].numel() for c in part)
            spans.append((x0, x1, y0, y1))

        def e2e_step():
            fork = torch.cuda.Event()
            fork.record(stream)
            copy_stream.wait_event(fork)
            arrived = []
            with torch.cuda.stream(copy_stream):
                for x0, x1, _, _ in spans:
                    X[x0:x1].copy_(HX[x0:x1], non_blocking=True)
                    e = torch.cuda.Event()
                    e.record(copy_stream)
                    arrived.append(e)
            done = []
            for (_, _, plan), e in zip(e2e_plans, arrived):
                stream.wait_event(e)
                plan.run(stream)
                d = torch.cuda.Event()
                d.record(stream)
                done.append(d)
            with torch.cuda.stream(copy_stream):
                for (_, _, y0, y1), d in zip(spans, done):
                    copy_stream.wait_event(d)
                    HY[y0:y1].copy_(Y[y0:y1], non_blocking=True)
            join = torch.cuda.Event()
            join.record(copy_stream)
            stream.wait_event(join)
    g = capture(e2e_step)
    e2e_reps = max(3, args.steps // 4)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    rank_barrier(world)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_reps):
            g.replay()
    torch.cuda.synchronize()
    te = max_over_ranks(time.perf_counter() - t0, world, device)
    del g
    e2e = {"value": round(whole_job_rate(wbytes, e2e_reps, world, te), 1), "unit": UNIT,
           "h2d_bytes_per_step": HX.numel() * 4, "d2h_bytes_per_step": HY.numel() * 4,
           "timing": ("host wall clock around CUDA-graph replays and the final sync; per launch group: its x in, "
                      "the launch, its y out, on a copy stream beside the compute stream" if batched else
                      "host wall clock around CUDA-graph replays (copy in, step, copy out) and the final sync")}

    cpu = None
    if rank == 0:
        v, cores, desc = time_oracle(host_sample, nv, budget_s=args.cpu_budget)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": desc}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "dtype_detail": "int8 x int8 -> int32 block sums, f32 block scales, f32 y",
        "data": "synthetic (seeded random GGUF blocks; x ~ N(0,1))",
        "config": {"workload": args.workload + ("" if args.layers in (None, 32) else f"[{args.layers} layers]"),
                   "n_vec": nv, "gemvs_per_step": len(calls),
                   "api": "qgemv_batched (one launch per type and row length)" if batched else "qgemv per matrix",
                   "weight_bytes_per_step": wbytes,
                   "l2": "inputs larger than L2 (weights rotate through distinct buffers > 4x L2)",
                   "timing": "CUDA graph of one step, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "hbm_frac": round(value / world / peak, 4), "hbm_peak_gbs": peak,
        "us_per_token": round(ms_per_step * 1e3, 2),
        "per_call": per_call, "breakdown": breakdown, "configs": configs,
        # dequantize_rows: timed on this workload's own weights for q4_k_4096,
        # else the figure the Q4_K 4096 x 4096 config above measured
        "dequantize_rows": dequant if dequant is not None else next(
            (dict(v["dequantize_rows"], workload=k) for k, v in (configs or {}).items()
             if isinstance(v, dict) and v.get("dequantize_rows")), None),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
    }
    return line


# ---------------------------------------------------------- reference arm
# --------------------------------------------------------- prefill workload
PREFILL = {"prefill_q4_k_4096": (12, 4096, 4096)}  # type id Q4_K, n_out, n_in


def run_prefill(args, rank, world, local_rank):
    """qgemm over n_tok tokens (default 512) on the library's default path
    (reported as config.plan): Q4_K expanded into tensor memory inside the
    GEMM, or W dequantized to f16 first. Value: the whole call's TFLOP/s
    (2 n_out n_in n_tok per call); roofline: the default path's GEMM against
    the measured tensor-core peak (the fused kernel together with the x
    conversion before it; the f16 GEMM alone through qgemm_f16)."""
    import torch

    import __graft_entry__
    import ggml_block_quantized_gb300 as qg
    from ggml_block_quantized_gb300 import synth

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    t, n_out, n_in = PREFILL[args.workload]
    n_tok = args.n_vec if args.n_vec > 8 else 512
    plan = qg.gemm_kernel_info(t, n_out, n_in, n_tok)  # the library's default routing and launches
    fused_default = plan.startswith("gemm_q4k_tmem_kernel")
    launches_per_call = int(plan.split("launches=")[1].split()[0])
    rng = np.random.default_rng(3000)
    Wh = synth.k_blocks(t, n_out * n_in // 256, rng)
    xh = synth.f32_normal(rng, n_tok * n_in)
    W0 = torch.from_numpy(Wh).to(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    copies = max(1, int(np.ceil(4 * l2 / W0.numel())))
    Ws = [W0] + [W0.clone() for _ in range(copies - 1)]
    X = torch.from_numpy(xh).to(device)
    Y = torch.empty((n_tok, n_out), dtype=torch.float32, device=device)
    ws = torch.empty(qg.qgemm_workspace_bytes(t, n_out, n_in, n_tok), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device)
    flops = 2.0 * n_out * n_in * n_tok

    def step():
        for W in Ws:
            qg.qgemm(t, W, X, n_out, n_in, n_tok, y=Y, workspace=ws, stream=stream)

    a_bytes = (2 * n_out * n_in + 255) // 256 * 256
    A16, B16 = ws[:2 * n_out * n_in], ws[a_bytes:a_bytes + 2 * n_tok * n_in]

    def gemm_only():
        for _ in Ws:
            qg.qgemm_f16(A16, B16, n_out, n_tok, n_in, y=Y, stream=stream)

    def graph(fn):
        with torch.cuda.stream(stream):
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    def timed(g, reps, sampler=None):
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup)):
                g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if sampler:
            sampler.start()
        rank_barrier(world)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        clocks = sampler.stop() if sampler else None
        return max_over_ranks(e0.elapsed_time(e1) / 1e3, world, device), clocks

    g = graph(step)
    sampler = ClockSampler(local_rank)
    tt, clocks = timed(g, args.steps, sampler)
    calls = args.steps * len(Ws)
    value = whole_job_rate(flops * len(Ws), args.steps, world, tt, 1e12)
    del g
    gg = graph(gemm_only)
    tg, _ = timed(gg, args.steps)
    del gg
    # the same calls with Q4_K dequantized inside the GEMM (no f16 copy of W),
    # and with the f16 copy of W (the default picks one by the token count)
    fused = {}
    for mode, where in ((1, "tensor memory"), (0, "an f16 copy in the workspace")):
        prev = qg.tune("QG_FUSED_GEMM", mode)
        try:
            gf = graph(step)
            tf, _ = timed(gf, args.steps)
            del gf
        finally:
            qg.tune("QG_FUSED_GEMM", prev)
        fused[f"QG_FUSED_GEMM={mode}"] = {
            "us_per_call": round(tf / calls * 1e6, 3),
            "TFLOP_s": round(whole_job_rate(flops * len(Ws), args.steps, world, tf, 1e12), 2),
            "note": (f"x to f16, then one GEMM that expands Q4_K blocks into {where}" if mode else
                     "W dequantized to an f16 copy and x to f16, then the GEMM")}
    gemm_us = tg / calls * 1e6
    achieved = flops / (tg / calls) / 1e12
    call_us = tt / calls * 1e6
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, peak_kind = float(json.load(f)["bf16_tflops"]), "measured (bf16 burst; f16 has the same nominal rate)"
    except Exception:
        peak, peak_kind = 1900.0, "fallback"
    assert qg.device_error() == 0, "a kernel reported a bounded-wait timeout"

    # end to end: x in from pinned host memory, y out, one call per step
    HX = X.cpu().pin_memory()
    HY = torch.empty(Y.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        X.copy_(HX, non_blocking=True)
        qg.qgemm(t, Ws[0], X, n_out, n_in, n_tok, y=Y, workspace=ws, stream=stream)
        HY.copy_(Y, non_blocking=True)
    ge = graph(e2e_step)
    reps = max(3, args.steps)
    with torch.cuda.stream(stream):
        ge.replay()
    torch.cuda.synchronize()
    rank_barrier(world)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(reps):
            ge.replay()
    torch.cuda.synchronize()
    te = max_over_ranks(time.perf_counter() - t0, world, device)
    del ge

    cpu = None
    if rank == 0:
        import oracle
        oracle.lib()
        rows = max(1, min(n_out, int(64 * args.cpu_budget)))
        t0 = time.perf_counter()
        oracle.gemm_float(t, Wh[:rows * n_in // 256 * 144], xh, rows, n_in, n_tok)
        tc = time.perf_counter() - t0
        cpu = {"value": round(2.0 * rows * n_in * n_tok / tc / 1e12, 6), "unit": "TFLOP/s",
               "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"{rows} of the {n_out} rows, all {n_tok} tokens (dequantize, f64 matmul)"}
    return {
        "metric": f"Q4_K prefill TFLOP/s ({n_out}x{n_in} weights, {n_tok} tokens; f16 operands, f32 accumulation)",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tt / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "dtype_detail": "W dequantized to f16, x rounded to f16, f32 accumulate",
        "data": "synthetic (seeded random Q4_K blocks; x ~ N(0,1))",
        "config": {"workload": args.workload, "n_tok": n_tok, "calls_per_step": len(Ws),
                   "api": ("qgemm (x to f16, tcgen05 GEMM expanding Q4_K blocks into tensor memory)" if fused_default
                           else "qgemm (dequantize to f16, x to f16, tcgen05 GEMM)"),
                   "plan": plan,
                   "l2": "weights rotate through distinct buffers > 4x L2",
                   "timing": "CUDA graph of one step, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "us_per_call": round(tt / calls * 1e6, 3), "fused_dequant": fused,
        # the default path's GEMM: the fused kernel cannot be timed apart from the
        # x conversion launched before it, so its entry is the whole call
        # (conversion included, an underestimate); the f16 GEMM is timed alone
        "roofline": ({"bound": "tensor", "kernel": plan.split()[0] + " with the x conversion before it (one qgemm call)",
                      "achieved": round(flops / (call_us * 1e-6) / 1e12, 1), "peak": peak, "peak_kind": peak_kind,
                      "unit": "TFLOP/s", "frac": round(flops / (call_us * 1e-6) / 1e12 / peak, 4),
                      "traffic": committed_traffic(f"{plan.split()[0]}@{args.workload}@{n_tok}", "gemm"),
                      "algorithmic_flops_per_launch": int(flops), "avg_launch_us": round(call_us, 3),
                      "launches": launches_per_call} if fused_default else
                     {"bound": "tensor", "kernel": "gemm_f16_tc_kernel, 128-row x 128- or 256-token tiles (qgemm_f16)",
                      "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind, "unit": "TFLOP/s",
                      "frac": round(achieved / peak, 4), "traffic": None,
                      "algorithmic_flops_per_launch": int(flops), "avg_launch_us": round(gemm_us, 3), "launches": 1}),
        "f16_gemm_alone": {"kernel": "gemm_f16_tc_kernel (qgemm_f16 on the f16 operands)", "us": round(gemm_us, 3),
                           "TFLOP_s": round(achieved, 1), "frac": round(achieved / peak, 4)},
        "cpu_baseline": cpu,
        "e2e": {"value": round(whole_job_rate(flops, reps, world, te, 1e12), 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": HX.numel() * 4, "d2h_bytes_per_step": HY.numel() * 4,
                "timing": "host wall clock around CUDA-graph replays (copy in, qgemm, copy out) and the final sync"},
        "gpu_launches": launches_per_call * calls, "clocks": clocks,
    }


def run_reference(args):
    """The oracle, as it stands, on the host cores: each step one bounded
    sample of the same workload; the metric is a rate, so a sample gives it."""
    import numpy as _np  # noqa: F401

    from ggml_block_quantized_gb300 import synth
    import oracle
    oracle.lib()
    if args.workload == "layer_stack":
        sample = [synth.layer_matrix(0, m, args.n_vec) for m in range(len(synth.LAYER_MATRICES))]
        for s in sample:
            s["W"] = s.pop("w_blocks")
    else:
        m = synth.single_matrix(args.workload, n_vec=args.n_vec)
        W = oracle.quantize(m["type"], m["w_f32"]) if "w_f32" in m else m["w_blocks"]
        sample = [dict(type=m["type"], n_out=m["n_out"], n_in=m["n_in"], W=W, x=m["x"])]
    per_step_budget = max(1.0, args.cpu_budget / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        time_oracle(sample[:1], args.n_vec, budget_s=per_step_budget)
    rates = []
    cores = 1
    desc = ""
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, cores, desc = time_oracle(sample, args.n_vec, budget_s=per_step_budget)
        rates.append(v)
    wall = time.perf_counter() - t0
    value = float(np.mean(rates))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded random GGUF blocks; x ~ N(0,1))",
        "config": {"workload": args.workload, "n_vec": args.n_vec},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="layer_stack",
                    choices=["layer_stack", "q8_0_256x1024", "q4_0_4096", "q4_k_4096", "q6_k_32000",
                             "q4_1_32000", "q5_0_32000", "q2_k_32000", "q3_k_32000", "q5_k_32000",
                             "prefill_q4_k_4096"])
    ap.add_argument("--n-vec", type=int, default=1)
    ap.add_argument("--e2e-head", type=int, default=8,
                    help="matrices in the end-to-end step's first launch (0: as many as the others)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle timing")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the other workloads measured beside the stack (configs object)")
    ap.add_argument("--layers", type=int, default=None,
                    help="decoder layers of the stack (default 32; fewer only for profiling captures)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.workload in PREFILL:
        line = run_prefill(args, rank, world, local_rank)
    else:
        line = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
