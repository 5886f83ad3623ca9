#!/usr/bin/env python
"""Benchmark of the selective-scan hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:
    causal conv1d+SiLU forward -> selective scan forward (with per-chunk checkpoints)
    -> selective scan backward (recompute from checkpoints) -> conv1d backward.
Metric: tokens/s (sequences x tokens per second) of that fwd+bwd step, and the achieved HBM
bandwidth of the scan kernels.  Default workload: the training-shaped Mamba-1 layer
(16 x 2048 tokens, d_inner 1536, d_state 16, d_conv 4, bf16 I/O, fp32 state, z gate and D
skip, checkpoints every 256 tokens).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME | --config I]
                        [--impl reference]
--config I picks the I-th workload of bwd_ssm_conv_gb300.workloads.WORKLOADS.
With N > 1 it is launched by torch.distributed.run, one process per GPU; each GPU runs an
independent replica (the path has no cross-GPU exchange), value = all tokens / max time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from bwd_ssm_conv_gb300.workloads import WORKLOADS, make_inputs, workload  # noqa: E402

METRIC = "selective-scan fwd+bwd tokens/s (B·L/s) and achieved HBM GB/s vs 8 TB/s"
DEFAULT_WORKLOAD = "mamba1_train_bf16_b16_l2048_d1536_n16"
SPEC_HBM_GBS = 8000.0


# ---- algorithmic bytes per token (what each stage must move at minimum) -------------------
def alg_bytes(w) -> dict:
    """Bytes per token each stage must read and write at minimum (activations in the I/O
    dtype, checkpoints fp32 every `chunk` tokens; parameters and states are negligible)."""
    io, D, H, N, G = w.io_bytes, w.channels, w.n_head, w.d_state, w.n_group
    zc = D if w.has_z else 0
    ck = 4.0 * D * N / w.chunk
    bc = 2 * G * N * io
    scan_fwd = (D + H + zc + D) * io + bc + ck                        # x, dt, z in; y out
    scan_bwd = (D + H + zc + D) * io + bc + ck + (D + H + zc) * io + bc  # + dy in; dx dt dz dB dC
    conv_fwd = 2 * D * io if w.d_conv else 0
    conv_bwd = 3 * D * io if w.d_conv else 0
    return {"conv_fwd": conv_fwd, "scan_fwd": scan_fwd, "scan_bwd": scan_bwd,
            "conv_bwd": conv_bwd}


# Algorithmic FP32 flops per (token, channel, state) element of the scan kernels (an FMA counts
# 2, a multiply 1; the SFU exponentials are counted separately).
#   forward:  delta*A (1), (delta x)*B (1), h = a h + u (2), y += C h (2)                    = 6
#   backward: two forward recomputes (4 each, without C h) + the adjoint: dh = gy C + carry (2),
#             dC += gy h (1), sum dh B (2), dB = dh delta x (1), carry = a dh (1),
#             w = carry h_prev (1), sum A w (2), dA += delta w (2), y_pre += C h (2)      = 22
# With one A per head (the Mamba-2 form) delta*A is one product per (token, head), not per
# element: 5 and 20.
SCAN_FLOPS = {"scan_fwd": 6, "scan_bwd": 22}
SCAN_FLOPS_SCALAR_A = {"scan_fwd": 5, "scan_bwd": 20}
FP32_LANES_PER_SM = 128   # measured: 128 FFMA lanes per SM per clock on GB300 (packed f32x2
                          # issues half the instructions at the same lane rate)


# DRAM traffic of the dominant kernel per launch, from one ncu capture of this workload
# (dram__bytes_read.sum + dram__bytes_write.sum; summary in profiles/).  Reported only while the
# kernel's sources hash to what was captured; any edit makes it null until it is captured again.
TRAFFIC_CAPTURES = {
    "scan_bwd": {
        "kernel": "scan_bwd_tma_kernel<bf16, persistent>",
        "bytes": 958956544 + 1293119744,
        "sources": {
            "bwd_ssm_conv_gb300/csrc/scan_bwd_tma.cu":
                "0592b6cd43bced5da92b596baa0b110a78e293c3cfe4de2dd02ac366981512fa",
            "bwd_ssm_conv_gb300/csrc/scan_bwd.cuh":
                "561a4c86d7706877ace6dfe08a6a6e6b2fec8fd6789769f1024dd61a739393f2",
            "bwd_ssm_conv_gb300/csrc/scan_common.cuh":
                "4a263de92c114f3b898a0bf7eb5949e3841f9132b66fa3ec99e15445b373861f",
        },
    },
}


def captured_traffic(stage: str):
    """(bytes, kernel) of the capture for `stage` if its sources are unchanged, else (None, None)."""
    cap = TRAFFIC_CAPTURES.get(stage)
    if cap is None:
        return None, None
    for rel, digest in cap["sources"].items():
        try:
            with open(os.path.join(ROOT, rel), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != digest:
                    return None, None
        except OSError:
            return None, None
    return cap["bytes"], cap["kernel"]


def _measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ---- clocks during the timed region ------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sel = [r for t, r in self.rows if t0 <= t <= t1] or [r for _, r in self.rows]
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in sel:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---- the step ----------------------------------------------------------------------------
def packed(specs, dev):
    """One flat device byte buffer holding tensors of the given (shape, dtype) specs at 256-byte
    aligned offsets; returns (buffer, views).  A step's inputs and its results each live in one
    such buffer, so that the end-to-end leg moves them with one copy per direction."""
    offs, off = [], 0
    for shape, dt in specs:
        nbytes = torch.Size(shape).numel() * torch.empty(0, dtype=dt).element_size()
        offs.append((off, nbytes))
        off = (off + nbytes + 255) // 256 * 256
    buf = torch.empty(max(off, 1), dtype=torch.uint8, device=dev)
    views = [buf[o:o + n].view(dt).view(shape) for (o, n), (shape, dt) in zip(offs, specs)]
    return buf, views


class Step:
    """Device buffers for one step of the hot path and the calls that run it."""

    def __init__(self, w, dev, inp):
        from bwd_ssm_conv_gb300 import binding as B
        self.B = B
        self.w = w
        self.dev = dev
        self.in_keys = [k for k in (["sx", "c"] if w.d_conv else ["x"]) +
                        ["dt", "A", "B", "C", "D", "z", "s0", "dy", "d_state_out"]
                        if inp.get(k) is not None]
        self.in_buf, views = packed([(inp[k].shape, inp[k].dtype) for k in self.in_keys], dev)
        d = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inp.items()
             if k not in self.in_keys}
        for k, v in zip(self.in_keys, views):
            v.copy_(inp[k])
            d[k] = v
        self.d = d
        ns, L, H, P, N = w.n_seqs, w.n_tok, w.n_head, w.head_dim, w.d_state
        io = w.torch_io
        f32 = torch.float32
        self.x = (torch.empty(ns, L, H * P, dtype=io, device=dev) if w.d_conv
                  else d["x"].view(ns, L, H * P))
        self.x4 = self.x.view(ns, L, H, P)
        # the step's results, in the order outputs() lists them, in one buffer
        ospec = [("y", (ns, L, H, P), io), ("st", (ns, H, P, N), f32)]
        if not w.fwd_only:
            ospec += [("d_sx", tuple(d["sx"].shape), io) if w.d_conv else ("d_x", (ns, L, H, P), io),
                      ("d_dt", tuple(d["dt"].shape), d["dt"].dtype),
                      ("d_A", tuple(d["A"].shape), f32), ("d_B", tuple(d["B"].shape), io),
                      ("d_C", tuple(d["C"].shape), io)]
            if d["D"] is not None:
                ospec.append(("d_D", tuple(d["D"].shape), f32))
            if d["z"] is not None:
                ospec.append(("d_z", (ns, L, H, P), io))
            if w.d_conv:
                ospec.append(("d_c", tuple(d["c"].shape), f32))
        self.out_buf, oviews = packed([(sh, dt) for _, sh, dt in ospec], dev)
        o = dict(zip([k for k, _, _ in ospec], oviews))
        self.y = o["y"]
        self.st = o["st"]
        nch = (L + w.chunk - 1) // w.chunk
        self.ck = torch.empty(ns, nch, H, P, N, dtype=f32, device=dev)
        shape = B.scan_shape(self.x4, d["dt"], d["A"], d["B"], d["s0"], w.chunk)
        self.ws_f = torch.empty(B.ssm_scan_workspace_size(shape, False), dtype=torch.uint8,
                                device=dev)
        self.ws_b = torch.empty(B.ssm_scan_workspace_size(shape, True), dtype=torch.uint8,
                                device=dev)
        if not w.fwd_only:
            self.g = dict(d_s0=torch.empty(ns, H, P, N, dtype=f32, device=dev),
                          d_x=o["d_x"] if "d_x" in o else torch.empty_like(self.x4),
                          d_dt=o["d_dt"], d_A=o["d_A"], d_B=o["d_B"], d_C=o["d_C"],
                          d_D=o.get("d_D"), d_z=o.get("d_z"), d_dt_bias=None)
        if w.d_conv and not w.fwd_only:
            self.ws_c = torch.empty(B.ssm_conv_workspace_size(ns, H * P, L, w.d_conv),
                                    dtype=torch.uint8, device=dev)
            self.d_sx = o["d_sx"]
            self.d_c = o["d_c"]

    def stages(self):
        B, w, d = self.B, self.w, self.d
        out = []
        if w.d_conv:
            out.append(("conv_fwd", lambda: B.ssm_conv_fwd(d["sx"], d["c"], None, silu=True,
                                                           out=self.x)))
        out.append(("scan_fwd", lambda: B.ssm_scan_fwd(
            self.x4, d["dt"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"], s0=d["s0"],
            chunk=w.chunk, ws=self.ws_f, out=(self.y, self.st, self.ck))))
        if not w.fwd_only:
            out.append(("scan_bwd", lambda: B.ssm_scan_bwd(
                self.x4, d["dt"], d["A"], d["B"], d["C"], d["dy"], D=d["D"], z=d["z"],
                s0=d["s0"], ckpt=self.ck, d_state_out=d["d_state_out"], chunk=w.chunk,
                ws=self.ws_b, out=self.g)))
            if w.d_conv:
                out.append(("conv_bwd", lambda: B.ssm_conv_bwd(
                    d["sx"], d["c"], self.g["d_x"].view(w.n_seqs, w.n_tok, w.channels), None,
                    silu=True, ws=self.ws_c, out=(self.d_sx, self.d_c, None))))
        return out

    def outputs(self):
        """The step's results a caller reads back (for the end-to-end leg)."""
        if self.w.fwd_only:
            return [self.y, self.st]
        res = [self.y, self.st, self.g["d_x"] if not self.w.d_conv else self.d_sx,
               self.g["d_dt"], self.g["d_A"], self.g["d_B"], self.g["d_C"]]
        for k in ("d_D", "d_z"):
            if self.g[k] is not None:
                res.append(self.g[k])
        if self.w.d_conv:
            res.append(self.d_c)
        return res

    def inputs(self):
        return [self.d[k] for k in self.in_keys]


def reduce_max(value: float, dist=None, device=None) -> float:
    """Max of a per-rank value over all ranks (the slowest replica sets the job's time)."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job tokens/s: every rank processes tokens_per_rank per step; weak scaling."""
    return world * tokens_per_rank / (ms_max * 1e-3)


def l2_flush_buffer(dev):
    props = torch.cuda.get_device_properties(dev)
    return torch.empty(2 * props.L2_cache_size // 4 + 1, dtype=torch.float32, device=dev)


def time_device(step, steps, warmup, flush):
    """Per-step CUDA-event times (ms) of the whole step and of each stage, on the stream the
    kernels are launched on; L2 flushed before every step (outside the timed events)."""
    stream = torch.cuda.current_stream()
    stages = step.stages()
    for _ in range(warmup):
        for _, fn in stages:
            fn()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)]
           for _ in range(steps)]
    from bwd_ssm_conv_gb300 import binding as B
    launches0 = B.ssm_kernel_launches()
    for i in range(steps):
        flush.zero_()
        evs[i][0].record(stream)
        for j, (_, fn) in enumerate(stages):
            fn()
            evs[i][j + 1].record(stream)
    launches = B.ssm_kernel_launches() - launches0
    torch.cuda.synchronize()
    total = [e[0].elapsed_time(e[-1]) for e in evs]
    per_stage = {name: [e[j].elapsed_time(e[j + 1]) for e in evs]
                 for j, (name, _) in enumerate(stages)}
    return total, per_stage, launches


def time_e2e_serial(step, steps, warmup):
    """Same step through the public API with host buffers, one stream: every step copies its
    inputs from pinned host memory, runs, and reads its results back before the next starts.
    Inputs and results each travel as one packed buffer (Step.in_buf / Step.out_buf)."""
    host_in = step.in_buf.cpu().pin_memory()
    host_out = torch.empty(step.out_buf.shape, dtype=torch.uint8, pin_memory=True)
    stages = step.stages()

    def one():
        step.in_buf.copy_(host_in, non_blocking=True)
        for _, fn in stages:
            fn()
        host_out.copy_(step.out_buf, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_e2e(pair, steps, warmup):
    """Same step through the public API with host buffers: every step copies all its inputs
    from pinned host memory and reads all its results back, each as one packed buffer (one
    copy per direction, so no per-tensor copy overhead).  Two device buffer sets (`pair`)
    and three streams let step i's kernels overlap the input copies of step i+1 and the result
    copies of step i-1; events keep each buffer set's copies and kernels in order.  Returns
    (ms per step from the first input copy to the last result copy, bytes in, bytes out)."""
    host_in = pair[0].in_buf.cpu().pin_memory()
    host_out = [torch.empty(st.out_buf.shape, dtype=torch.uint8, pin_memory=True) for st in pair]
    stages = [st.stages() for st in pair]
    h2d = host_in.numel()
    d2h = host_out[0].numel()
    s_in, s_run, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    run_done, out_done = [None, None], [None, None]

    def one(i):
        k = i % 2
        with torch.cuda.stream(s_in):
            if run_done[k] is not None:  # step i-2's kernels are done with this input set
                s_in.wait_event(run_done[k])
            pair[k].in_buf.copy_(host_in, non_blocking=True)
            in_done = torch.cuda.Event()
            in_done.record(s_in)
        with torch.cuda.stream(s_run):
            s_run.wait_event(in_done)
            if out_done[k] is not None:  # step i-2's results have left this output set
                s_run.wait_event(out_done[k])
            for _, fn in stages[k]:
                fn()
            run_done[k] = torch.cuda.Event()
            run_done[k].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(run_done[k])
            host_out[k].copy_(pair[k].out_buf, non_blocking=True)
            out_done[k] = torch.cuda.Event()
            out_done[k].record(s_out)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(warmup, warmup + steps):
        one(i)
    e1.record(s_out)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


# ---- the oracle on the host (CPU baseline and the reference arm) ---------------------------
def config_of(w, world: int) -> dict:
    """The workload description both arms print."""
    return {"workload": w.name, "n_seqs": w.n_seqs, "seq_len": w.n_tok, "d_inner": w.channels,
            "head_dim": w.head_dim, "d_state": w.d_state, "d_conv": w.d_conv, "chunk": w.chunk,
            "state_dtype": "f32", "parallelism": f"replicas{world}",
            "l2": "flushed before every step"}


def oracle_sample(w, channels, seqs=1, seed=None):
    """Runs the oracle's whole step on `seqs` sequences x all tokens x `channels` channels of
    the workload; returns (seconds, channel-tokens processed)."""
    import oracle
    inp = make_inputs(w.with_(n_seqs=seqs, n_head=channels), seed=seed)
    t0 = time.perf_counter()
    dims = oracle.ScanDims(seqs, w.n_tok, channels, w.head_dim, w.d_state, n_group=w.n_group,
                           a_per_state=0 if w.scalar_a else 1, chunk=w.chunk)
    if w.d_conv:
        x = oracle.conv_fwd(inp["sx"], inp["c"], None, silu=True)
        x = x.reshape(seqs, w.n_tok, channels, w.head_dim)
    else:
        x = inp["x"]
    _, _, ck = oracle.scan_fwd(dims, x=x, dt=inp["dt"], A=inp["A"], B=inp["B"], C=inp["C"],
                               D=inp["D"], z=inp["z"], s0=inp["s0"])
    if not w.fwd_only:
        g = oracle.scan_bwd(dims, x=x, dt=inp["dt"], A=inp["A"], B=inp["B"], C=inp["C"],
                            dy=inp["dy"], D=inp["D"], z=inp["z"], ckpt=ck)
        if w.d_conv:
            oracle.conv_bwd(inp["sx"], inp["c"], g["d_x"].reshape(seqs, w.n_tok, channels),
                            silu=True)
    return time.perf_counter() - t0, seqs * w.n_tok * channels


def cpu_baseline(w, budget_s=12.0):
    """Oracle tokens/s at the workload's full width, from a bounded sample of the workload:
    whole sequences of all channels when they fit the budget, else a channel subset."""
    t, ct = oracle_sample(w, channels=4 * w.head_dim if w.head_dim > 1 else 4)
    per_ct = t / ct
    full_seq = per_ct * w.n_tok * w.n_head  # seconds for one sequence, all channels
    if full_seq <= budget_s:
        seqs = max(1, min(w.n_seqs, int(budget_s / full_seq)))
        ch = w.n_head
    else:
        seqs, ch = 1, max(1, int(budget_s / (per_ct * w.n_tok)))
    t, ct = oracle_sample(w, channels=ch, seqs=seqs)
    tokens_per_s = ct / t / w.n_head  # every channel of every token
    return {"value": tokens_per_s, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{seqs} of {w.n_seqs} sequences x {w.n_tok} tokens x {ch} of {w.n_head} "
                      f"channels of the same workload, full step (conv fwd, scan fwd, scan bwd, "
                      f"conv bwd), {t:.1f} s single-threaded f64; scaled to all channels"}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # size each step so that warmup + steps finish in about two minutes
    t, ct = oracle_sample(w, channels=2)
    per_ct = t / ct
    budget = 120.0 / max(1, args.steps + args.warmup)
    ch = max(1, min(w.n_head, int(budget / (per_ct * w.n_tok))))
    for _ in range(args.warmup):
        oracle_sample(w, channels=ch)
    times = [oracle_sample(w, channels=ch)[0] for _ in range(args.steps)]
    t_mean = sum(times) / len(times)
    value = (ch * w.n_tok / t_mean) / w.n_head
    sample = (f"each step: 1 sequence x {w.n_tok} tokens x {ch} of {w.n_head} channels, full "
              f"step, single-threaded f64 oracle; tokens/s scaled to all channels")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * w.n_seqs * w.n_tok / value, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[x.name for x in WORKLOADS])
    ap.add_argument("--config", type=int, default=None,
                    help="position of the workload in WORKLOADS (overrides --workload)")
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = WORKLOADS[args.config] if args.config is not None else workload(args.workload)
    if args.impl == "reference":
        run_reference(args, w)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from bwd_ssm_conv_gb300.build import build
    if rank == 0 or world == 1:
        build()
    if dist is not None:
        dist.barrier()

    inp = make_inputs(w, grad_seed_state=False)
    step = Step(w, dev, inp)
    flush = l2_flush_buffer(dev)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    total, per_stage, launches = time_device(step, args.steps, args.warmup, flush)
    t_wall1 = time.time()
    clocks = sampler.stop(t_wall0, t_wall1)
    ms = reduce_max(sum(total) / len(total), dist, dev)
    if dist is not None:
        dist.barrier()

    e2e_steps = max(3, min(args.steps, 20))
    serial_ms = reduce_max(time_e2e_serial(step, e2e_steps, 2), dist, dev)
    e2e_ms, h2d, d2h = time_e2e((step, Step(w, dev, inp)), e2e_steps, 2)
    e2e_ms = reduce_max(e2e_ms, dist, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    tokens = w.n_seqs * w.n_tok
    value = job_throughput(tokens, world, ms)
    peaks, peak_src = _measured_peaks()
    ab = alg_bytes(w)
    stage_ms = {k: sum(v) / len(v) for k, v in per_stage.items()}
    dom = max(stage_ms, key=stage_ms.get)
    dom_bytes = ab[dom] * tokens
    achieved = dom_bytes / (stage_ms[dom] * 1e-3) / 1e9
    stage_gbs = {k: ab[k] * tokens / (stage_ms[k] * 1e-3) / 1e9 for k in stage_ms}
    props = torch.cuda.get_device_properties(dev)
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
    fp32_peak = props.multi_processor_count * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12  # TFLOP/s
    traffic, traffic_kernel = captured_traffic(dom)
    if dom in SCAN_FLOPS:
        # The scan kernels are bound by FP32 arithmetic, not HBM: per element the backward needs
        # ~22 flops for ~0.9 bytes, far above the GB300 ridge (~12 flops/byte).
        elems = tokens * w.channels * w.d_state
        flops = (SCAN_FLOPS_SCALAR_A if w.scalar_a else SCAN_FLOPS)[dom] * elems
        ach_tf = flops / (stage_ms[dom] * 1e-3) / 1e12
        roofline = {"kernel": f"ssm_{dom}", "bound": "alu", "achieved": ach_tf,
                    "peak": fp32_peak, "unit": "TFLOP/s", "frac": ach_tf / fp32_peak,
                    "peak_source": f"derived: SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 x {mhz:.0f} MHz",
                    "traffic": traffic, "traffic_kernel": traffic_kernel,
                    "algorithmic_flops_per_launch": flops,
                    "hbm": {"achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                            "frac": achieved / peaks["hbm_gbs"], "peak_source": peak_src,
                            "algorithmic_bytes_per_launch": dom_bytes}}
    else:
        roofline = {"kernel": f"ssm_{dom}", "bound": "hbm", "achieved": achieved,
                    "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                    "peak_source": peak_src, "traffic": traffic, "traffic_kernel": traffic_kernel,
                    "algorithmic_bytes_per_launch": dom_bytes}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.io == "bf16" else "f32", "data": "synthetic",
        "config": config_of(w, world),
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "stage_hbm_gbs": {k: round(v, 1) for k, v in stage_gbs.items()},
        "stage_frac_of_8tbs": {k: round(v / SPEC_HBM_GBS, 4) for k, v in stage_gbs.items()},
        "roofline": roofline,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "e2e": {"value": job_throughput(tokens, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipelined": "2 buffer sets, copies of steps i+1 / i-1 overlap step i; inputs and results each one packed copy",
                "serial_ms_per_step": serial_ms},
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
