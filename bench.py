"""Benchmark of the block-sparse attention backward (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload w1|w4|...]
    python bench.py --impl reference ...      # the fp64 CPU oracle, same metric

A step is one bsa_grad call (mask compaction, preprocess, tcgen05 backward,
finalize) over the workload's inputs, already resident in HBM. The L2 is
flushed (a 512 MB write) between timed steps; each step is timed with CUDA
events on the launching stream. FLOPs are the algorithmic 10*bx*by*D per
active block per query head. Under torchrun every rank runs its own replica
of the workload on its GPU (no data-path collective); the step time is the
max over ranks and `value` counts the work of all ranks.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-sparse attn bwd TFLOP/s (active blocks) & % of GB300 BF16 tensor peak"
UNIT = "TFLOP/s"
FALLBACK_PEAK = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}


LAUNCHES_PER_STEP = 7  # kernels of one bsa_grad call

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="w1")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations timed after the default w1 line")
    ap.add_argument("--config-steps", type=int, default=100,
                    help="timed steps of each other configuration")
    ap.add_argument("--key-block64", action="store_true",
                    help="blockShape [bx, 64] workloads: one query-major step per 64-key block")
    ap.add_argument("--deterministic", action="store_true",
                    help="time the deterministic dQ mode (separate query-tile pass)")
    ap.add_argument("--forward", action="store_true",
                    help="time the companion forward (bsa_fwd) instead of the backward")
    return ap.parse_args()


def dist_setup(n):
    import torch
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAK, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_hash():
    """The backward kernel's sources and those of its work plan (planner
    kernel, host planning), which set the kernel's memory traffic too."""
    h = hashlib.sha256()
    for f in ("bsa_bwd.cu", "sm103_ptx.cuh", "bsa_kernels.cu", "bsa_api.cpp"):
        with open(os.path.join(ROOT, "block_sparse_attention_attn_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def committed_traffic(workload):
    """DRAM bytes per launch of the backward kernel from the committed ncu
    summary, or None when the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "bwd_kernel_counters.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("source_hash") != kernel_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ inputs
def torch_dtype(name):
    import torch
    return {"bf16": torch.bfloat16, "f16": torch.float16}[name]


def make_inputs(w, dev):
    import torch

    import block_sparse_attention_attn_gb300 as bsa
    dt = torch_dtype(w.dtype)
    dout, q, k, v = (torch.from_numpy(x).to(dt).to(dev) for x in w.tensors())
    mask = None if w.mask is None else torch.from_numpy(w.mask).to(dev)
    am = None if w.atten_mask is None else torch.from_numpy(w.atten_mask).to(dev)
    seq = dict(actual_seq_lengths=w.seq_q, actual_seq_lengths_kv=w.seq_kv)
    out, lse, fws = bsa.block_sparse_attention_fwd(q, k, v, block_sparse_mask=mask,
                                                 block_shape=[w.bx, w.by], layout=w.layout,
                                                 num_key_value_heads=w.N2, scale_value=w.scale,
                                                 atten_mask=am, **seq, **w.window_kw())
    bsa.bsa_check_status(fws)
    return dict(dout=dout, query=q, key=k, value=v, attention_out=out, softmax_lse=lse,
                block_sparse_mask=mask, atten_mask=am), seq


DETERMINISTIC = False  # set from --deterministic
KEY_BLOCK64 = False    # set from --key-block64


def grad_executor(w, t, seq, dq, dk, dv):
    import block_sparse_attention_attn_gb300 as bsa
    size, ex = bsa.bsa_grad_workspace_size(
        t["dout"], t["query"], t["key"], t["value"], t["attention_out"], t["softmax_lse"],
        t["block_sparse_mask"], t["atten_mask"], [w.bx, w.by], seq["actual_seq_lengths"],
        seq["actual_seq_lengths_kv"], w.layout, w.layout, w.N2,
        0 if t["atten_mask"] is None else 1, w.scale, w.pre_tokens, w.next_tokens,
        dq=dq, dk=dk, dv=dv)
    if DETERMINISTIC:
        ex.set_deterministic(True)
    if KEY_BLOCK64:
        ex.set_key_block64(True)
    return size, ex


# --------------------------------------------------------------- our arm
def time_backward(w, t, seq, dq, dk, dv, steps, warmup, local, world):
    """The timed protocol of one workload: `warmup` untimed steps, then
    `steps` steps, each after a 512 MB L2 flush, bracketed by CUDA events on
    the launching stream (the step time); then the same number of steps again
    with the library's own events around the main kernel (the kernel time: the
    two event records inside the call add about 5 us to a step, so they stay
    out of the pass that gives the step time). Returns (mean step ms, mean
    kernel ms, clocks, wall s of the first pass, ws, size)."""
    import torch

    import block_sparse_attention_attn_gb300 as bsa
    dev = dq.device
    size, ex = grad_executor(w, t, seq, dq, dk, dv)
    ws = torch.empty(size, dtype=torch.uint8, device=dev)
    del ex
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(ex, ev=None):
        if ev is not None:
            ex.set_timing_events(*ev)
        bsa.bsa_grad(ws, size, ex, stream)

    for _ in range(warmup):
        flush.zero_()
        step(grad_executor(w, t, seq, dq, dk, dv)[1])
    torch.cuda.synchronize()
    bsa.bsa_check_status(ws)

    n = steps
    # host-side planning (first stage) happens before the timed region
    exs = [grad_executor(w, t, seq, dq, dk, dv)[1] for _ in range(2 * n)]
    s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    k0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    k1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in k0 + k1:
        e.record(stream)   # materialise the event handles before handing them to C
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    wall0 = time.perf_counter()
    for i in range(n):
        flush.zero_()
        s_ev[i].record(stream)
        step(exs[i])
        e_ev[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    for i in range(n):
        flush.zero_()
        step(exs[n + i], (k0[i], k1[i]))
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    bsa.bsa_check_status(ws)
    del flush
    step_ms = [a.elapsed_time(b) for a, b in zip(s_ev, e_ev)]
    kern_ms = [a.elapsed_time(b) for a, b in zip(k0, k1)]
    ms_step = max_over_ranks(float(np.mean(step_ms)), world)
    ms_kern = max_over_ranks(float(np.mean(kern_ms)), world)
    return ms_step, ms_kern, clk, wall, ws, size


def e2e_pipelined(t, outs, size_of, launch, n_steps):
    """End-to-end time per step through the public API: every step copies
    its inputs (the device tensors of dict `t`) from pinned host memory to the
    device, runs both stages of the library call (`size_of(inputs, outputs)`
    gives the workspace size, `launch(inputs, outputs, ws, size, stream)` runs
    the first and second stage) and reads the outputs `outs` back into pinned
    host memory. The inputs sit packed in one pinned host buffer and, per
    buffer set, one device buffer (the outputs likewise), so each direction is
    one copy per step; two device buffer sets alternate, and the copies run on
    their own streams, so the host-to-device copy of step i+1 and the
    read-back of step i-1 overlap the compute of step i. Returns (ms per step, H2D bytes,
    D2H bytes per step), timed with CUDA events from the first copy to the
    last read-back."""
    import torch

    import block_sparse_attention_attn_gb300 as bsa
    compute = torch.cuda.current_stream()
    dev = outs[0].device

    def layout(tensors):
        """Byte offsets of the tensors packed back to back (256-byte aligned)."""
        offs, off = [], 0
        for x in tensors:
            offs.append(off)
            off += (x.numel() * x.element_size() + 255) // 256 * 256
        return offs, max(off, 256)

    def carve(flat, like, off):
        n = like.numel() * like.element_size()
        return flat[off:off + n].view(like.dtype).view(like.shape)

    # the inputs packed in one pinned host buffer and, per buffer set, one
    # device buffer, so each step moves its inputs with one copy and its
    # outputs with one read-back
    names = [k_ for k_, x in t.items() if x is not None]
    in_offs, in_bytes = layout([t[k_] for k_ in names])
    out_offs, out_bytes = layout(outs)
    h_in = torch.empty(in_bytes, dtype=torch.uint8, pin_memory=True)
    for k_, off in zip(names, in_offs):
        carve(h_in, t[k_], off).copy_(t[k_].cpu())
    sets = []
    for k in range(2):
        d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        d_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        ti = {k_: None for k_ in t}
        for k_, off in zip(names, in_offs):
            ti[k_] = carve(d_in, t[k_], off)
        oi = tuple(carve(d_out, x, off) for x, off in zip(outs, out_offs))
        d_in.copy_(h_in)
        size = size_of(ti, oi)
        ws = torch.empty(max(size, 256), dtype=torch.uint8, device=dev)
        h_out = torch.empty(out_bytes, dtype=torch.uint8, pin_memory=True)
        sets.append((ti, oi, ws, size, d_in, d_out, h_out))
    h2d = sum(t[k_].numel() * t[k_].element_size() for k_ in names)
    d2h = sum(x.numel() * x.element_size() for x in outs)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_c = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def run(i):
        k = i % 2
        ti, oi, ws, size, d_in, d_out, h_out = sets[k]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_c[k])      # step i-2 has read this set's inputs
            d_in.copy_(h_in, non_blocking=True)
            ev_in[k].record(s_in)
        compute.wait_event(ev_in[k])
        if i >= 2:
            compute.wait_event(ev_out[k])     # step i-2's outputs have been read back
        launch(ti, oi, ws, size, compute)
        ev_c[k].record(compute)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_c[k])
            h_out.copy_(d_out, non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(2):                        # warm-up
        run(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(compute)
    s_in.wait_event(start)
    for i in range(2, 2 + n_steps):
        run(i)
    compute.wait_stream(s_out)                # after the last read-backs
    end.record(compute)
    torch.cuda.synchronize()
    for st_ in sets:
        bsa.bsa_check_status(st_[2])
    return start.elapsed_time(end) / n_steps, h2d, d2h




# The other configurations of the workload table, timed in the same run
# after the headline one (w1dense: the w1 shape with mask = nullptr).
# (record name, workload, mode): mode "grad" is the default backward, "det"
# the deterministic dQ mode, "k64" the 64-key-block kernel, "fwd" the forward
OTHER_CONFIGS = [("w1dense", "w1dense", "grad"), ("w2", "w2", "grad"), ("w3", "w3", "grad"),
                 ("w4", "w4", "grad"), ("w3_key_block64", "w3", "k64"),
                 ("w1_deterministic", "w1", "det"), ("w4_deterministic", "w4", "det"),
                 ("w1_forward", "w1", "fwd"), ("w4_forward", "w4", "fwd")]


def other_configs(args, world, local, peak):
    """kernel / step time, roofline fraction and clocks of OTHER_CONFIGS."""
    import torch

    import block_sparse_attention_attn_gb300 as bsa
    from block_sparse_attention_attn_gb300.workloads import make_workload
    global DETERMINISTIC, KEY_BLOCK64
    dev = torch.device("cuda", local)
    res = {}
    saved = (DETERMINISTIC, KEY_BLOCK64)
    for key, name, mode in OTHER_CONFIGS:
        w = make_workload(name)
        flops = (0.4 if mode == "fwd" else 1.0) * w.flops()
        t, seq = make_inputs(w, dev)
        steps = max(3, min(args.steps, args.config_steps))
        if mode == "fwd":
            q, k, v = t["query"], t["key"], t["value"]
            out, lse = torch.empty_like(t["attention_out"]), torch.empty_like(t["softmax_lse"])

            def fwd_executor():
                return bsa.bsa_fwd_workspace_size(
                    q, k, v, t["block_sparse_mask"], [w.bx, w.by], seq["actual_seq_lengths"],
                    seq["actual_seq_lengths_kv"], w.layout, w.layout, w.N2, w.scale,
                    w.pre_tokens, w.next_tokens, out, lse, t["atten_mask"])
            ms_step, ms_kern, clk = time_forward(fwd_executor, steps, max(3, args.warmup),
                                                 local, world)
            del q, k, v, out, lse
        else:
            DETERMINISTIC, KEY_BLOCK64 = mode == "det", mode == "k64"
            dq, dk, dv = (torch.empty_like(t[k_]) for k_ in ("query", "key", "value"))
            ms_step, ms_kern, clk, _, ws, _ = time_backward(w, t, seq, dq, dk, dv, steps,
                                                            max(3, args.warmup), local, world)
            DETERMINISTIC, KEY_BLOCK64 = saved
            del dq, dk, dv, ws
        ach = flops / (ms_kern * 1e-3) / 1e12
        res[key] = {"workload": name, "mode": {"grad": "default backward",
                                               "det": "backward, deterministic dQ",
                                               "k64": "backward, 64-key blocks",
                                               "fwd": "companion forward (4*D FLOP per pair)"}[mode],
                    "gflop_per_step": round(flops / 1e9, 2), "steps": steps,
                    "ms_per_step": round(ms_step, 4),
                    "value": round(world * flops / (ms_step * 1e-3) / 1e12, 2),
                    "kernel_ms": round(ms_kern, 4), "achieved": round(ach, 2),
                    "frac": round(ach / peak, 4),
                    "traffic": committed_traffic(name) if mode == "grad" else None,
                    "clocks": clk}
        del t
        torch.cuda.empty_cache()
    DETERMINISTIC, KEY_BLOCK64 = saved
    return res


def bench_ours(args, rank, world, local):
    import torch

    import block_sparse_attention_attn_gb300 as bsa
    from block_sparse_attention_attn_gb300.workloads import make_workload, workload_summary
    dev = torch.device("cuda", local)
    w = make_workload(args.workload)
    flops = w.flops()
    t, seq = make_inputs(w, dev)
    dq = torch.empty_like(t["query"])
    dk = torch.empty_like(t["key"])
    dv = torch.empty_like(t["value"])
    n = args.steps
    ms_step, ms_kern, clk, wall, ws, size = time_backward(w, t, seq, dq, dk, dv, n, args.warmup,
                                                          local, world)
    value = world * flops / (ms_step * 1e-3) / 1e12

    # end to end through the public API: pinned host inputs -> H2D -> first and
    # second stage -> D2H of dq, dk, dv, every step (copies of one step overlap
    # the compute of the previous one)
    e2e_ms, h2d, d2h = e2e_pipelined(
        t, (dq, dk, dv), lambda ti, o: grad_executor(w, ti, seq, *o)[0],
        lambda ti, o, ws, size, st: bsa.bsa_grad(ws, size, grad_executor(w, ti, seq, *o)[1], st),
        max(3, min(n, 20)))
    e2e_ms = max_over_ranks(e2e_ms, world)

    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAK["bf16_tflops"]))
    achieved = flops / (ms_kern * 1e-3) / 1e12
    summ = workload_summary(w)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded PCG64 N(0,1) inputs; Out/lse from bsa_fwd)",
        "config": {"workload": w.name, "layout": w.layout, "B": w.B, "N1": w.N1, "N2": w.N2,
                   "Sq": w.Sq, "Skv": w.Skv, "D": w.D, "block": [w.bx, w.by],
                   "active_blocks": summ["active_blocks"], "density": round(summ["density"], 4),
                   "gflop_per_step": round(flops / 1e9, 2), "parallelism": f"replicas x{world}",
                   "l2": "flushed (512 MB write) before every timed step",
                   "dq_mode": "deterministic (query-tile pass)" if DETERMINISTIC else "fp32 reduce-add",
                   "key_block64": KEY_BLOCK64 and w.by == 64 and w.D == 128 and not w.token_masked(),
                   "window": ([w.pre_tokens, w.next_tokens] if w.windowed() else None),
                   "atten_mask": (w.atten_mask_desc or None)},
        "pct_of_peak": round(100.0 * value / world / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "traffic": None if DETERMINISTIC else committed_traffic(w.name),
                     "kernel": ("k_bwd + k_bwd_dq (tcgen05 backward, deterministic dQ)"
                                if DETERMINISTIC else "k_bwd (tcgen05 backward)"),
                     "kernel_ms": round(ms_kern, 4),
                     "kernel_timing": "CUDA events around the kernel on its stream, in a "
                                      "second pass of the same number of flushed steps",
                     "peak_source": f"{src}: MEASURED_PEAKS.json bf16_tflops (burst)"
                     if src == "measured" else "fallback 1.9 PFLOP/s bf16"},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "schedule": "inputs and outputs packed (one copy each way per step); two device "
                            "buffer sets; the H2D copy of step i+1 and the D2H "
                            "read-back of step i-1 run on copy streams during step i"},
        # per step: info upload, mask compaction (count, fill), planner,
        # preprocess, backward, finalize
        "gpu_launches": LAUNCHES_PER_STEP * n,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
    }
    if args.workload == "w1" and not args.no_configs:
        line["configs"] = other_configs(args, world, local, peak)
    if not args.no_cpu_baseline and rank == 0:
        try:
            line["cpu_baseline"] = cpu_baseline(w)
        except Exception as exc:  # the GPU numbers stand on their own
            line["cpu_baseline"] = {"value": None, "unit": UNIT, "cores": os.cpu_count(),
                                    "kind": "oracle", "sample": f"failed: {exc!r}"}
    return line


# ------------------------------------------------- companion forward arm
FWD_METRIC = "block-sparse attn fwd TFLOP/s (companion forward, active blocks)"


def time_forward(fwd_executor, steps, warmup, local, world):
    """The timed protocol of the forward (as time_backward's): `warmup`
    untimed steps, then `steps` steps, each after a 512 MB L2 flush, with CUDA
    events around the call, then as many with events around the main kernel.
    Returns (mean step ms, mean kernel ms, clocks)."""
    import torch

    import block_sparse_attention_attn_gb300 as bsa
    size, _ = fwd_executor()
    ws = torch.empty(size, dtype=torch.uint8, device=torch.cuda.current_device())
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=ws.device)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush.zero_()
        bsa.bsa_fwd(ws, size, fwd_executor()[1], stream)
    torch.cuda.synchronize()
    bsa.bsa_check_status(ws)
    n = steps
    exs = [fwd_executor()[1] for _ in range(2 * n)]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for e in ev:
        e[1].record(stream)
        e[2].record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.2)
    for i in range(n):
        flush.zero_()
        ev[i][0].record(stream)
        bsa.bsa_fwd(ws, size, exs[i], stream)
        ev[i][3].record(stream)
    for i in range(n):
        flush.zero_()
        exs[n + i].set_timing_events(ev[i][1], ev[i][2])
        bsa.bsa_fwd(ws, size, exs[n + i], stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    bsa.bsa_check_status(ws)
    ms_step = max_over_ranks(float(np.mean([e[0].elapsed_time(e[3]) for e in ev])), world)
    ms_kern = max_over_ranks(float(np.mean([e[1].elapsed_time(e[2]) for e in ev])), world)
    del flush
    return ms_step, ms_kern, clk


def bench_forward(args, rank, world, local):
    """The same protocol for bsa_fwd: Out and lse of one workload per step;
    4*D FLOP per (query, key) pair per query head (S = QK^T and O = PV)."""
    import torch

    import block_sparse_attention_attn_gb300 as bsa
    from block_sparse_attention_attn_gb300.workloads import make_workload
    dev = torch.device("cuda", local)
    w = make_workload(args.workload)
    flops = 0.4 * w.flops()
    t, seq = make_inputs(w, dev)
    q, k, v = t["query"], t["key"], t["value"]
    out, lse = torch.empty_like(t["attention_out"]), torch.empty_like(t["softmax_lse"])

    def fwd_executor():
        return bsa.bsa_fwd_workspace_size(
            q, k, v, t["block_sparse_mask"], [w.bx, w.by], seq["actual_seq_lengths"],
            seq["actual_seq_lengths_kv"], w.layout, w.layout, w.N2, w.scale, w.pre_tokens,
            w.next_tokens, out, lse, t["atten_mask"])

    n = args.steps
    ms_step, ms_kern, clk = time_forward(fwd_executor, n, args.warmup, local, world)
    # end to end: pinned host Q, K, V (and masks) -> H2D -> both stages -> D2H of Out, lse
    fin = {k_: t[k_] for k_ in ("query", "key", "value", "block_sparse_mask", "atten_mask")}

    def fwd_size(ti, o):
        return bsa.bsa_fwd_workspace_size(
            ti["query"], ti["key"], ti["value"], ti["block_sparse_mask"], [w.bx, w.by],
            seq["actual_seq_lengths"], seq["actual_seq_lengths_kv"], w.layout, w.layout, w.N2,
            w.scale, w.pre_tokens, w.next_tokens, o[0], o[1], ti["atten_mask"])

    e2e_ms, h2d, d2h = e2e_pipelined(
        fin, (out, lse), lambda ti, o: fwd_size(ti, o)[0],
        lambda ti, o, ws, size, st: bsa.bsa_fwd(ws, size, fwd_size(ti, o)[1], st),
        max(3, min(n, 20)))
    e2e_ms = max_over_ranks(e2e_ms, world)
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAK["bf16_tflops"]))
    achieved = flops / (ms_kern * 1e-3) / 1e12
    line = {
        "metric": FWD_METRIC, "value": round(world * flops / (ms_step * 1e-3) / 1e12, 2),
        "unit": UNIT, "n_gpus": world, "steps": n, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded PCG64 N(0,1) inputs)",
        "config": {"workload": w.name, "pass": "forward", "gflop_per_step": round(flops / 1e9, 2),
                   "parallelism": f"replicas x{world}",
                   "l2": "flushed (512 MB write) before every timed step",
                   "window": ([w.pre_tokens, w.next_tokens] if w.windowed() else None),
                   "atten_mask": (w.atten_mask_desc or None)},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "k_fwd (tcgen05 forward)", "kernel_ms": round(ms_kern, 4),
                     "kernel_timing": "CUDA events around the kernel on its stream, in a "
                                      "second pass of the same number of flushed steps",
                     "peak_source": f"{src}: MEASURED_PEAKS.json bf16_tflops (burst)"
                     if src == "measured" else "fallback 1.9 PFLOP/s bf16"},
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "schedule": "inputs and outputs packed (one copy each way per step); two device "
                            "buffer sets; the H2D copy of step i+1 and the D2H "
                            "read-back of step i-1 run on copy streams during step i"},
        "gpu_launches": (3 if w.atten_mask is not None else 2) * n,  # info upload, [mask packing,] forward
        "clocks": clk,
    }
    if not args.no_cpu_baseline and rank == 0:
        from oracle import bsa_oracle as O
        S = min(w.Sq, 2048)
        a, kw, fl = _oracle_sample(w, 1, S)
        t0 = time.perf_counter()
        O.forward(a[1], a[2], a[3], **kw)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": round(0.4 * fl / dt / 1e12, 6), "unit": UNIT,
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{w.name} batch 0, 1 query head, first {S} tokens "
                                          f"({0.4 * fl / 1e9:.2f} GFLOP, {dt:.1f} s)"}
    return line


# ------------------------------------------------------- CPU oracle timings
def _oracle_sample(w, heads, S):
    """The workload restricted to batch 0, the first `heads` query heads (and
    their key heads) and the first S tokens; returns (args, kwargs, flops)."""
    import torch
    dt = torch_dtype(w.dtype)   # same rounding as the GPU inputs
    G = w.N1 // w.N2
    g_heads = -(-heads // G)
    rng = np.random.Generator(np.random.PCG64(w.seed + 99))
    def rnd(n):
        return torch.from_numpy(rng.standard_normal((1, n, S, w.D), dtype=np.float32) * w.std) \
            .to(dt).to(torch.float64).numpy()
    q, dout, out = rnd(heads), rnd(heads), rnd(heads) * 0.1
    k, v = rnd(g_heads), rnd(g_heads)
    from block_sparse_attention_attn_gb300.workloads import Workload
    mask = None if w.mask is None else w.mask[:1, :heads, :-(-S // w.bx), :-(-S // w.by)]
    lse = np.full((1, heads, S, 1), math.log(S) + 2.0)
    am = None if w.atten_mask is None else w.atten_mask[:S, :S]
    kw = dict(mask=mask, block_shape=(w.bx, w.by), num_kv_heads=g_heads, scale=w.scale,
              atten_mask=am, **w.window_kw())
    sample = Workload(w.name, "BNSD", w.dtype, 1, heads, g_heads, w.D, w.bx, w.by, [S], [S], S, S,
                      w.scale, mask, atten_mask=am, **w.window_kw())
    return (dout, q, k, v, out, lse), kw, sample.flops()


def cpu_baseline(w, target_s=12.0):
    """The oracle (fp64 numpy, as it stands) on a bounded sample of the workload:
    batch 0, the first S <= 4096 tokens, as many query heads as fit in about
    `target_s` seconds, repeated until that much CPU time has passed."""
    from oracle import bsa_oracle as O
    S = min(w.Sq, 4096)
    args, kw, fl = _oracle_sample(w, 1, S)
    t0 = time.perf_counter()
    O.backward(*args, **kw)
    dt = time.perf_counter() - t0
    heads = max(1, min(w.N1, int(target_s / max(dt, 1e-3))))
    args, kw, fl = _oracle_sample(w, heads, S)
    reps, total = 0, 0.0
    while total < target_s * 0.8 or reps == 0:
        t0 = time.perf_counter()
        O.backward(*args, **kw)
        total += time.perf_counter() - t0
        reps += 1
    return {"value": round(reps * fl / total / 1e12, 6), "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{w.name} batch 0, {heads} query heads, first {S} tokens, same mask, "
                      f"{reps} run(s) ({fl / 1e9:.1f} GFLOP algorithmic each, {total:.1f} s "
                      f"in total, numpy fp64 BLAS threads)"}


def bench_reference(args, rank, world):
    from block_sparse_attention_attn_gb300.workloads import make_workload
    from oracle import bsa_oracle as O
    w = make_workload(args.workload)
    S = min(w.Sq, 1024)
    a, kw, fl = _oracle_sample(w, 1, S)
    for _ in range(args.warmup):
        O.backward(*a, **kw)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        O.backward(*a, **kw)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * float(np.mean(times))
    value = fl / (ms * 1e-3) / 1e12
    sample = f"{w.name} batch 0, 1 query head, first {S} tokens, same mask ({fl / 1e9:.2f} GFLOP)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample": sample},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if rank != 0:
            return
        print(json.dumps(bench_reference(args, rank, world)), flush=True)
        return
    global DETERMINISTIC, KEY_BLOCK64
    DETERMINISTIC = args.deterministic
    KEY_BLOCK64 = args.key_block64
    rank, world, local = dist_setup(args.gpus)
    line = (bench_forward if args.forward else bench_ours)(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
