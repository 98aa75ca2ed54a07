"""Benchmark of the grouped expert MLP (forward + input gradient) on GB300.

One step = one pass of the whole expert path over one batch: permute, grouped
FC1 with fused SwiGLU, grouped FC2, weighted combine, then the output-gradient
permute, dgrad FC2 with fused SwiGLU backward, dgrad FC1 and the dX combine.
Default workload: the balanced 128-expert layer (E=128, H=2048, F=768,
T=16384 tokens, top-8, uniform routing), synthetic seeded data.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gg|reference]

With N > 1 (launched by torch.distributed.run) every rank runs an independent
replica of the step on its own GPU (the path has no exchange step here), and
rank 0 prints the whole-job line: units of all ranks / max-over-ranks time.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_synth import CONFIGS, make_inputs  # noqa: E402

METRIC = "expert-MLP fwd+dgrad TFLOP/s & tokens/s on 1 GB300; % BF16 tensor peak"
DEFAULT_CFG = 2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


# ------------------------------------------------------------------ captured DRAM traffic

_CSRC = os.path.join(ROOT, "moe_expert_grouped_gb300", "csrc")
TRAFFIC_FILES = {
    "bf16": os.path.join(ROOT, "profiles", "gemm_dram_traffic_balanced_e128_t16384.md"),
    "mxfp8": os.path.join(ROOT, "profiles", "gemm_mx_dram_traffic_balanced_e128_t16384.md"),
}
GEMM_SOURCES = {
    "bf16": [os.path.join(_CSRC, f) for f in ("gg_gemm.cu", "gg_epilogue.cuh", "gg_ptx.cuh",
                                              "gg_internal.h")],
    "mxfp8": [os.path.join(_CSRC, f) for f in ("gg_gemm_mx.cu", "gg_mx.cuh", "gg_epilogue.cuh",
                                               "gg_ptx.cuh", "gg_internal.h")],
}


def gemm_sources_sha256(precision: str = "bf16") -> str:
    import hashlib

    h = hashlib.sha256()
    for f in GEMM_SOURCES[precision]:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def captured_traffic(op: str, workload: str, precision: str = "bf16"):
    """DRAM bytes (read + write) per launch of `op` from the committed ncu
    summary, or None when there is none for this workload or the GEMM sources
    changed since it was captured."""
    path = TRAFFIC_FILES[precision]
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            line = line.strip().lstrip("-").strip()
            if ":" in line:
                key, _, val = line.partition(":")
                fields[key.strip().strip("`")] = val.strip().strip("`")
    if fields.get("sources_sha256") != gemm_sources_sha256(precision):
        return None
    if fields.get("workload") != workload:
        return None
    try:
        return int(fields[f"{op}_dram_bytes"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ multi-rank plumbing

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_seconds: float, local_units: float, backend_device=None):
    """(max seconds over ranks, sum of units over ranks); identity without a process group."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return local_seconds, local_units
    dev = backend_device if backend_device is not None else torch.device("cpu")
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.window = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(device_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        """Stop sampling; the summary of the window given to mark()."""
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return self.summary(self.window)

    def summary(self, window):
        """Median SM clock, max clock and active throttle reasons of the
        samples inside `window` (all samples when none fell inside it)."""
        if self.proc is None:
            return None
        inside = [s for t, s in list(self.samples) if window and window[0] <= t <= window[1]]
        used = inside if inside else [s for _, s in list(self.samples)]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[0]) for s in used if num(s[0]) is not None]
        mx = [num(s[1]) for s in used if num(s[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in used for i in range(4) if s[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples_in_window": len(inside), "samples": len(self.samples)}


# ------------------------------------------------------------------ oracle timing

def time_oracle(shape, inp, n_tokens: int, steps: int = 1, **variant):
    """Wall time of the fp64 oracle forward + input and probability gradients on a
    token sample."""
    import oracle

    sel = np.arange(min(n_tokens, shape.T))
    W1 = oracle.bf16_bits_to_f64(inp.W1)  # the oracle's documented fp64 weight form
    W2 = oracle.bf16_bits_to_f64(inp.W2)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        fwd = oracle.moe_forward(inp.x[sel], inp.idx[sel], inp.prob[sel], W1, W2, shape.E, shape.P,
                                 **variant)
        oracle.moe_backward(inp.dOut[sel], fwd, W1, W2)
        times.append(time.perf_counter() - t0)
    return times, sel.size


def blas_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001
        pass
    return os.cpu_count()


# ------------------------------------------------------------------ the gg arm

def run_gg(args, shape, peaks):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    import moe_expert_grouped_gb300.gg as gg

    inp = make_inputs(shape, 1000 * args.config + 17 * rank)

    def to_dev(u16):
        return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(dev)

    x, dOut = to_dev(inp.x), to_dev(inp.dOut)
    W1, W2 = to_dev(inp.W1), to_dev(inp.W2)
    idx = torch.from_numpy(inp.idx).to(dev)
    prob = torch.from_numpy(inp.prob).to(dev)
    T, H, F, k, E, P = shape.T, shape.H, shape.F, shape.k, shape.E, shape.P
    act = {"swiglu": gg.GG_ACT_SWIGLU, "qgeglu": gg.GG_ACT_QGEGLU}[args.activation]
    mode = {"combine": gg.GG_PROB_COMBINE, "activation": gg.GG_PROB_ACTIVATION,
            "pre_fc1": gg.GG_PROB_PRE_FC1}[args.prob_mode]
    epi_f = gg.GG_EPI_QGEGLU if act == gg.GG_ACT_QGEGLU else gg.GG_EPI_SWIGLU
    epi_b = gg.GG_EPI_QGEGLU_BWD if act == gg.GG_ACT_QGEGLU else gg.GG_EPI_SWIGLU_BWD
    pre = mode == gg.GG_PROB_PRE_FC1
    rec = args.recompute_h1
    mx = args.precision == "mxfp8"
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    dX = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    dprob = torch.empty((T, k), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    if mx:
        # the frozen weights are quantised once, outside the timed region
        mxw, _ = gg.mx_prepare_weights(W1, W2)
        layer = gg.MxMoeLayer(T, H, F, k, E, P, device=dev, activation=act, prob_mode=mode)
        b = {n: layer.view(n) for n in gg.MxMoeLayer._SHAPES}
        ops = ["permute", "quant_x", "fc1_swiglu", "fc2", "combine", "quant_dout",
               "dgrad_fc2_swiglu_bwd", "dgrad_fc1", "combine_dx"]

        def run_layer(x_, idx_, prob_, dO_, o_, dX_, dp_):
            layer.forward(x_, idx_, prob_, mxw, out=o_)
            layer.backward(dO_, mxw, dX=dX_, dprob=dp_)
    else:
        layer = gg.MoeLayer(T, H, F, k, E, P, device=dev, activation=act, prob_mode=mode,
                            recompute_h1=rec)
        b = {n: layer.view(n) for n in ("Xp", "H1", "A", "Yp", "dYp", "dH", "dXp", "offsets",
                                        "row_of_slot", "slot_of_row", "prob_of_row", "rowdot",
                                        "ws")}
        ops = ["permute", "fc1_swiglu", "fc2", "combine", "permute_dout",
               "dgrad_fc2_swiglu_bwd", "dgrad_fc1", "combine_dx"]
        if rec:
            ops.insert(4, "fc1_recompute")

        def run_layer(x_, idx_, prob_, dO_, o_, dX_, dp_):
            layer.forward(x_, idx_, prob_, W1, W2, out=o_)
            layer.backward(dO_, W1, W2, dX=dX_, dprob=dp_)
    ws = b["ws"]
    rc = layer.R_cap

    def step_mx(events=None):
        # the same calls, in the same order, as gg_moe_mlp_fwd_mx + gg_moe_mlp_bwd_mx
        def mark(i):
            if events is not None:
                events[i].record(stream)

        por = b["prob_of_row"]
        nt = int(layer.buf.n_tiles)
        mark(0)
        gg.permute(x, idx, prob, E, P, ws=ws, out=dict(b, Xp=None))
        mark(1)
        gg.mx_quantize_rows(x, b, k, E, P, ws, prob=prob if pre else None, n_tiles=nt,
                            out=dict(Q=b["Xq"], S=b["Xs"], tiles_before=b["tiles_before"]))
        mark(2)
        gg.mx_grouped_gemm(gg.GG_MX_FC1, b["Xq"], b["Xs"], mxw, b["offsets"], E, rc, H, F, ws,
                           activation=act, Cq=b["Aq"], Cs=b["As"], H1=b["H1"],
                           row_scale=por if mode == gg.GG_PROB_ACTIVATION else None)
        mark(3)
        gg.mx_grouped_gemm(gg.GG_MX_FC2, b["Aq"], b["As"], mxw, b["offsets"], E, rc, H, F, ws,
                           activation=act, C=b["Yp"])
        mark(4)
        gg.unpermute_combine(b["Yp"], b["row_of_slot"], prob if mode == gg.GG_PROB_COMBINE else None,
                             T, k, ws, out=out)
        mark(5)
        gg.mx_quantize_rows(dOut, b, k, E, P, ws, n_tiles=nt,
                            out=dict(Q=b["dYq"], S=b["dYs"], tiles_before=b["tiles_before"]))
        mark(6)
        gg.mx_grouped_gemm(gg.GG_MX_DGRAD_FC2, b["dYq"], b["dYs"], mxw, b["offsets"], E, rc, H, F,
                           ws, activation=act, Cq=b["dHq"], Cs=b["dHs"], H1=b["H1"],
                           row_scale=None if pre else por,
                           rowdot=b["rowdot"] if mode == gg.GG_PROB_ACTIVATION else None)
        mark(7)
        gg.mx_grouped_gemm(gg.GG_MX_DGRAD_FC1, b["dHq"], b["dHs"], mxw, b["offsets"], E, rc, H, F,
                           ws, activation=act, C=b["dXp"])
        mark(8)
        if pre:
            gg.unpermute_combine(b["dXp"], b["row_of_slot"], prob, T, k, ws, out=dX, dprob=dprob,
                                 dot_src=x)
        elif mode == gg.GG_PROB_COMBINE:
            gg.unpermute_combine_dot(b["dXp"], b["row_of_slot"], None, T, k, dOut, b["Yp"], ws,
                                     out=dX, dprob=dprob)
        else:
            gg.unpermute_combine(b["dXp"], b["row_of_slot"], None, T, k, ws, out=dX,
                                 rowdot=b["rowdot"], dprob=dprob,
                                 n_rowdot=gg.mx_rowdot_blocks(F))
        mark(9)

    def step(events=None):
        # the same calls, in the same order, as gg_moe_mlp_fwd + gg_moe_mlp_bwd
        def mark(i):
            if events is not None:
                events[i].record(stream)

        mark(0)
        if pre:  # row maps, then the copy that takes the probability along
            gg.permute(x, idx, prob, E, P, ws=ws, out=dict(b, Xp=None))
            gg.permute_rows(x, b["row_of_slot"], b["slot_of_row"], b["offsets"], k, E, P, rc, ws,
                            dst=b["Xp"], prob=prob)
        else:
            gg.permute(x, idx, prob, E, P, ws=ws, out=b)
        mark(1)
        gg.grouped_fwd(b["Xp"], W1, b["offsets"], epi_f, ws=ws, C=b["A"],
                       H1_save=None if rec else b["H1"],
                       prob_of_row=b["prob_of_row"] if mode == gg.GG_PROB_ACTIVATION else None)
        mark(2)
        gg.grouped_fwd(b["A"], W2, b["offsets"], gg.GG_EPI_NONE, ws=ws, C=b["Yp"])
        mark(3)
        gg.unpermute_combine(b["Yp"], b["row_of_slot"], prob if mode == gg.GG_PROB_COMBINE else None,
                             T, k, ws, out=out)
        mark(4)
        i = 4
        if rec:  # the backward's recompute of FC1's output (a plain grouped FC1)
            gg.grouped_fwd(b["Xp"], W1, b["offsets"], gg.GG_EPI_NONE, ws=ws, C=b["H1"])
            i += 1
            mark(i)
        gg.permute_rows(dOut, b["row_of_slot"], b["slot_of_row"], b["offsets"], k, E, P, rc, ws,
                        dst=b["dYp"])
        mark(i + 1)
        gg.grouped_dgrad(b["dYp"], W2, b["offsets"], epi_b, H1=b["H1"],
                         prob_of_row=None if pre else b["prob_of_row"], ws=ws, dA=b["dH"],
                         rowdot=None if pre else b["rowdot"])
        mark(i + 2)
        gg.grouped_dgrad(b["dH"], W1, b["offsets"], gg.GG_EPI_NONE, ws=ws, dA=b["dXp"])
        mark(i + 3)
        if pre:
            gg.unpermute_combine(b["dXp"], b["row_of_slot"], prob, T, k, ws, out=dX, dprob=dprob,
                                 dot_src=x)
        else:
            gg.unpermute_combine(b["dXp"], b["row_of_slot"], None, T, k, ws, out=dX,
                                 rowdot=b["rowdot"], dprob=dprob, n_rowdot=gg.rowdot_blocks(F))
        mark(i + 4)

    if mx:
        step = step_mx  # noqa: F811
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if gg.read_status(ws) != 0:
        raise RuntimeError("device status after warm-up: " + gg.status_string(gg.read_status(ws)))

    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler is not None:
        time.sleep(0.5)  # let nvidia-smi start producing samples
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ops) + 1)]
          for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n0 = gg.launch_count()
    wall0 = time.time()
    start.record(stream)
    for s in range(args.steps):
        step(ev[s])
    end.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    launches = gg.launch_count() - n0
    if world > 1:
        dist.barrier()
    if sampler is not None:
        sampler.mark(wall0, wall1)
    local_s = start.elapsed_time(end) / 1e3
    status = gg.read_status(ws)
    if status != 0:
        raise RuntimeError("device status after timing: " + gg.status_string(status))

    per_op = {op: [ev[s][i].elapsed_time(ev[s][i + 1]) for s in range(args.steps)]
              for i, op in enumerate(ops)}
    flop_step = shape.flop_fwd() + shape.flop_dgrad()
    tot_s, tot_flop = aggregate(local_s, flop_step * args.steps,
                                dev if world > 1 else None)
    _, tot_tokens = aggregate(local_s, float(T * args.steps), dev if world > 1 else None)

    # ---- end to end through the public API with host buffers (pinned)
    # Every step copies its inputs host->device and its results device->host
    # inside the timed region. The copies run on two copy streams with two
    # device buffer sets, so step s+1's inputs arrive and step s-1's results
    # leave while step s computes (a streaming caller's pipeline).
    h_x = torch.from_numpy(inp.x.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_dO = torch.from_numpy(inp.dOut.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_idx = torch.from_numpy(inp.idx).pin_memory()
    h_prob = torch.from_numpy(inp.prob).pin_memory()
    h_out = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h_dX = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h_dp = [torch.empty((T, k), dtype=torch.float32).pin_memory() for _ in range(2)]
    d_in = [(torch.empty_like(x), torch.empty_like(idx), torch.empty_like(prob),
             torch.empty_like(dOut)) for _ in range(2)]
    d_res = [(torch.empty_like(out), torch.empty_like(dX), torch.empty_like(dprob))
             for _ in range(2)]
    s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set i landed
    ev_used = [torch.cuda.Event() for _ in range(2)]   # compute done with set i
    ev_out = [torch.cuda.Event() for _ in range(2)]    # results of set i copied out

    def e2e_run(n_steps):
        for i in range(2):
            ev_used[i].record(stream)
            ev_out[i].record(stream)
        for s in range(n_steps):
            i = s & 1
            dx_, didx_, dprob_, ddO_ = d_in[i]
            with torch.cuda.stream(s_h2d):
                s_h2d.wait_event(ev_used[i])
                dx_.copy_(h_x, non_blocking=True)
                didx_.copy_(h_idx, non_blocking=True)
                dprob_.copy_(h_prob, non_blocking=True)
                ddO_.copy_(h_dO, non_blocking=True)
                ev_in[i].record(s_h2d)
            o_, dX_, dp_ = d_res[i]
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_out[i])
            run_layer(dx_, didx_, dprob_, ddO_, o_, dX_, dp_)
            ev_used[i].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(ev_used[i])
                h_out[i].copy_(o_, non_blocking=True)
                h_dX[i].copy_(dX_, non_blocking=True)
                h_dp[i].copy_(dp_, non_blocking=True)
                ev_out[i].record(s_d2h)
        for i in range(2):
            stream.wait_event(ev_out[i])

    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_s, _ = aggregate(e0.elapsed_time(e1) / 1e3, 0.0, dev if world > 1 else None)
    if gg.read_status(layer.view("ws")) != 0:
        raise RuntimeError("device status after the end-to-end run")
    if not (torch.equal(h_out[0], out.cpu()) and torch.equal(h_dX[0], dX.cpu())
            and torch.equal(h_dp[0], dprob.cpu())):
        raise RuntimeError("end-to-end results differ from the device-resident step")
    h2d = x.numel() * 2 + dOut.numel() * 2 + idx.numel() * 4 + prob.numel() * 4
    d2h = out.numel() * 2 + dX.numel() * 2 + dprob.numel() * 4

    # ---- sustained: at least --sustained-s seconds of back-to-back steps
    # after the timed region and the end-to-end run, with their own clock
    # record (a seconds-long training step runs the layer under the power
    # cap, not as a burst)
    sus = None
    if args.sustained_s > 0:
        n_sus = max(args.steps, int(args.sustained_s / max(local_s / args.steps, 1e-6)) + 1)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        sw0 = time.time()
        s0.record(stream)
        for _ in range(n_sus):
            step()
        s1.record(stream)
        torch.cuda.synchronize(dev)
        sw1 = time.time()
        sus_s, _ = aggregate(s0.elapsed_time(s1) / 1e3, 0.0, dev if world > 1 else None)
        if gg.read_status(ws) != 0:
            raise RuntimeError("device status after the sustained run")
        sus = {"steps": n_sus, "seconds": round(sus_s, 3), "window": (sw0, sw1)}


    clocks = sampler.stop() if sampler is not None else None
    if sus is not None:
        sus["clocks"] = sampler.summary(sus.pop("window")) if sampler is not None else None
        sus.pop("window", None)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    # ---- roofline of the dominant kernel
    rc = layer.R_cap

    def hbm_bytes(op):
        # algorithmic bytes: permute reads idx/prob and writes the row maps;
        # the combines read k rows per token (+ row map, prob) and write one
        # (MXFP8: the permute writes the row maps only, the row quantisers
        # read each token row once and write one E4M3 row + scales per pair)
        quant = T * H * 2 + R * H + R * H // 32 + 4 * R
        return {"permute": (8 * R + 4 * R + 8 * rc) + (0 if mx else (T + R) * H * 2),
                "permute_dout": (T + R) * H * 2 + 4 * rc,
                "quant_x": quant, "quant_dout": quant,
                "combine": (R + T) * H * 2 + 8 * R,
                # MXFP8 with the probability at the combine: the dX combine also
                # reads the kept Yp rows and dOut for the probability gradient
                "combine_dx": (R + T) * H * 2 + 4 * R + (
                    (R + T) * H * 2 if mx and mode == gg.GG_PROB_COMBINE else 0)}[op]

    avg = {op: float(np.mean(v)) for op, v in per_op.items()}
    total_ms = sum(avg.values())
    R = shape.R
    # (with --recompute-h1 the backward's FC1 recompute is extra work the
    # metric does not count: `value` stays 12·R·H·F per step)
    flop_of = {"fc1_swiglu": 4.0 * R * H * F, "fc2": 2.0 * R * H * F,
               "dgrad_fc2_swiglu_bwd": 2.0 * R * H * F, "dgrad_fc1": 4.0 * R * H * F,
               "fc1_recompute": 4.0 * R * H * F}
    dom = max(avg, key=lambda o: avg[o])
    # MXFP8 contractions run at twice the BF16 rate (nominal 4.5 vs 2.25 PFLOP/s
    # dense): their peak is the measured BF16 burst times that ratio
    tensor_peak = peaks["bf16_tflops"] * (2.0 if mx else 1.0)
    tensor_src = f"{peaks['source']} bf16 burst" + (" x 2 (nominal fp8/bf16 ratio)" if mx else "")
    if dom in flop_of:
        ach = flop_of[dom] / (avg[dom] / 1e3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": round(ach, 2),
                "peak": round(tensor_peak, 1), "unit": "TFLOP/s",
                "frac": round(ach / tensor_peak, 4),
                "traffic": captured_traffic(dom, shape.name, args.precision),
                "peak_source": tensor_src}
    else:
        byts = hbm_bytes(dom)
        ach = byts / (avg[dom] / 1e3) / 1e9
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4),
                "traffic": None, "peak_source": f"{peaks['source']} hbm copy"}
    hbm_ops = {op: hbm_bytes(op) for op in ops if op not in flop_of}
    kernels = {}
    for op in ops:
        entry = {"ms": round(avg[op], 4), "share": round(avg[op] / total_ms, 4)}
        if op in flop_of:
            entry["tflops"] = round(flop_of[op] / (avg[op] / 1e3) / 1e12, 1)
        else:
            entry["gbs"] = round(hbm_ops[op] / (avg[op] / 1e3) / 1e9, 1)
        kernels[op] = entry

    # ---- CPU baseline: the oracle on a bounded token sample (rank 0, N = 1)
    cpu = None
    if world == 1 and not args.no_cpu_baseline and not mx:
        times, n_tok = time_oracle(shape, inp, args.cpu_tokens, activation=args.activation,
                                   prob_mode=args.prob_mode)
        sub = shape.with_tokens(n_tok)
        cpu_val = (sub.flop_fwd() + sub.flop_dgrad()) / times[0] / 1e12
        cpu = {"value": cpu_val, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"{n_tok} of {T} tokens (all k slots), numpy fp64 forward + input "
                         f"and probability gradients, {times[0]:.2f} s, "
                         f"tokens/s {n_tok / times[0]:.1f}"}

    value = tot_flop / tot_s / 1e12

    def per_ghz(v, clk):
        mhz = (clk or {}).get("sm_mhz")
        return round(v / world / (mhz / 1e3), 2) if mhz else None

    sustained = None
    if sus is not None:
        sus_value = flop_step * sus["steps"] * world / sus["seconds"] / 1e12
        sustained = {"value": round(sus_value, 2), "unit": "TFLOP/s",
                     "steps": sus["steps"], "seconds": sus["seconds"],
                     "ms_per_step": round(sus["seconds"] / sus["steps"] * 1e3, 4),
                     "tokens_per_s": round(T * sus["steps"] * world / sus["seconds"], 1),
                     "pct_vs_2250_tflops": round(sus_value / world / 2250.0, 4),
                     "tflops_per_ghz": per_ghz(sus_value, sus["clocks"]),
                     "clocks": sus["clocks"]}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "mxfp8" if mx else "bf16",
        "data": "synthetic",
        "config": {"workload": shape.name, "E": E, "H": H, "F": F, "T": T, "k": k, "P": P,
                   "routing": shape.routing, "parallelism": f"replicas x{world}",
                   "outputs": "out, dX, dprob", "activation": args.activation,
                   "prob_mode": args.prob_mode, "recompute_h1": rec,
                   "precision": args.precision,
                   "l2": "inputs larger than L2 (weights 1.2 GB, activations > 1 GB per step)"},
        "tokens_per_s": round(tot_tokens / tot_s, 1),
        "pct_bf16_peak": {"vs_2250_tflops": round(value / world / 2250.0, 4),
                          "vs_measured_burst": round(value / world / peaks["bf16_tflops"], 4),
                          "vs_measured_sustained": round(
                              value / world / peaks["bf16_tflops_sustained"], 4)},
        "roofline": roof, "kernels": kernels,
        "e2e": {"value": round(tot_flop / e2e_s / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "tokens_per_s": round(T * args.steps * world / e2e_s, 1)},
        "gpu_launches": int(launches), "clocks": clocks, "cpu_baseline": cpu,
        "launches_per_step": int(launches) // max(1, args.steps),
        "tflops_per_ghz": per_ghz(value, clocks),
        "sustained": sustained,
    }
    if mx:
        line["pct_fp8_peak"] = {"vs_4500_tflops": round(value / world / 4500.0, 4),
                                "vs_measured_bf16_burst_x2": round(
                                    value / world / (2 * peaks["bf16_tflops"]), 4)}
        line["cpu_baseline_note"] = ("the oracle's MXFP8 layer quantises every expert's weights "
                                     "in fp64; the timed CPU baseline is on the BF16 line")
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return line


# ------------------------------------------------------------------ the reference arm

def run_reference(args, shape):
    world, rank, _ = dist_env()
    if rank != 0:
        return None  # the oracle runs once, on rank 0's host cores
    inp = make_inputs(shape, 1000 * args.config)
    import oracle

    W1 = oracle.bf16_bits_to_f64(inp.W1)
    W2 = oracle.bf16_bits_to_f64(inp.W2)
    n = min(args.ref_tokens, shape.T)
    rng = np.random.default_rng(0)

    def step():
        sel = np.sort(rng.choice(shape.T, size=n, replace=False))
        fwd = oracle.moe_forward(inp.x[sel], inp.idx[sel], inp.prob[sel], W1, W2, shape.E, shape.P,
                                 activation=args.activation, prob_mode=args.prob_mode)
        oracle.moe_backward(inp.dOut[sel], fwd, W1, W2)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    sub = shape.with_tokens(n)
    flop = (sub.flop_fwd() + sub.flop_dgrad()) * args.steps
    value = flop / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": shape.name, "E": shape.E, "H": shape.H, "F": shape.F,
                   "T": shape.T, "k": shape.k, "P": shape.P, "routing": shape.routing,
                   "parallelism": "host cores", "outputs": "out, dX, dprob",
                   "activation": args.activation, "prob_mode": args.prob_mode},
        "tokens_per_s": n * args.steps / dt,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"{n} random tokens of {shape.T} per step (all k slots), "
                                   "numpy fp64 forward + input and probability gradients"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return line


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gg", "reference"], default="gg")
    ap.add_argument("--config", type=int, default=DEFAULT_CFG, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--tokens", type=int, default=0, help="override T (sweep points)")
    ap.add_argument("--cpu-tokens", type=int, default=8192)
    ap.add_argument("--ref-tokens", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustained-s", type=float, default=2.0,
                    help="seconds of back-to-back steps timed after the timed region "
                         "(0: none)")
    ap.add_argument("--activation", choices=["swiglu", "qgeglu"], default="swiglu")
    ap.add_argument("--recompute-h1", action="store_true",
                    help="do not keep FC1's output for the backward; recompute it there")
    ap.add_argument("--prob-mode", choices=["combine", "activation", "pre_fc1"],
                    default="combine", help="where the routing probability is applied")
    ap.add_argument("--precision", choices=["bf16", "mxfp8"], default="bf16",
                    help="bf16: the frozen BF16 weights; mxfp8: MXFP8 operands on the "
                         "block-scaled tensor cores (weights quantised once, untimed)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.precision == "mxfp8" and args.recompute_h1:
        ap.error("--recompute-h1 is a BF16 option")
    shape = CONFIGS[args.config]
    if args.tokens:
        shape = shape.with_tokens(args.tokens)
    if args.impl == "reference":
        return run_reference(args, shape)
    return run_gg(args, shape, load_peaks())


if __name__ == "__main__":
    main()
