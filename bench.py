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
    # the fused calls read sx where the scan reads x and write d_sx where it writes dx
    return {"conv_fwd": conv_fwd, "scan_fwd": scan_fwd, "scan_bwd": scan_bwd,
            "conv_bwd": conv_bwd, "conv_scan_fwd": scan_fwd, "conv_scan_bwd": scan_bwd}


# Algorithmic FP32 flops per (token, channel, state) element of the method itself (an FMA
# counts 2, a multiply 1; the SFU exponentials are counted separately), for the secondary ALU
# view of the roofline:
#   forward:  delta*A (1), (delta x)*B (1), h = a h + u (2), y += C h (2)                    = 6
#   backward: one recompute of the state (4, as the forward without C h) and the adjoint:
#             dh = gy C + carry (2), carry = a dh (1), w = carry h_prev (1), dA += delta w (2),
#             sum A w (2), sum dh B (2), dB += dh delta x (2), dC += gy h (2), y_pre += C h (2)
#                                                                                          = 20
# With one A per head (the Mamba-2 form) delta*A is one product per (token, head): 5 and 19.
SCAN_FLOPS = {"scan_fwd": 6, "scan_bwd": 20}
SCAN_FLOPS_SCALAR_A = {"scan_fwd": 5, "scan_bwd": 19}
FP32_LANES_PER_SM = 128   # measured: 128 FFMA lanes per SM per clock on GB300 (packed f32x2
                          # issues half the instructions at the same lane rate)
# The two configurations the throughput target is stated on; the default run measures both.
TARGET_WORKLOADS = ("mamba1_long_bf16_b1_l16384_d2048_n16", DEFAULT_WORKLOAD)


# DRAM traffic of the dominant kernel per launch, from one ncu capture of this workload
# (dram__bytes_read.sum + dram__bytes_write.sum; summary in profiles/).  Reported only while the
# kernel's sources hash to what was captured; any edit makes it null until it is captured again.
TRAFFIC_CAPTURES = {
    "scan_bwd": {
        "kernel": "scan_bwd_tma_kernel<bf16, persistent>",
        "bytes": 461442560 + 361737728,
        "sources": {
            "bwd_ssm_conv_gb300/csrc/scan_bwd_tma.cu":
                "50f08915816a813e680fc1512b7a4133b49d337a81fdf7ecb2442007c3afc24e",
            "bwd_ssm_conv_gb300/csrc/scan_bwd.cuh":
                "1ba6a1c2e1acc8aa74133a18acf8163297c25c51b3485aade9655a20773ec648",
            "bwd_ssm_conv_gb300/csrc/scan_common.cuh":
                "ec33325a539666d13bd9bd7e0e477eef67041e67e6335846b2a0d300e8def98a",
            "bwd_ssm_conv_gb300/csrc/tmem.cuh":
                "a55a9f2b432aed93c2a879bdb73a942f1e4300594365b99509ffbe376fc332f5",
            "bwd_ssm_conv_gb300/csrc/tma.cuh":
                "7faa420ff2e14fc905e7e16a643798cbd631d272b9772c9e1d3e1d9fbd4b4f6c",
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
    """Device buffers for one step of the hot path and the calls that run it.  path "split":
    ssm_conv_fwd -> ssm_scan_fwd -> ssm_scan_bwd -> ssm_conv_bwd, x kept between the forward
    and the backward; "fused": ssm_conv_scan_fwd -> ssm_conv_scan_bwd, x never stored by the
    forward (the backward recomputes it)."""

    def __init__(self, w, dev, inp, path="split"):
        from bwd_ssm_conv_gb300 import binding as B
        self.B = B
        self.w = w
        self.dev = dev
        self.path = path if w.d_conv else "split"
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
        if self.path == "fused":
            csh = B.conv_scan_shape(d["sx"], d["c"], d["dt"], d["A"], d["B"], d["s0"], w.chunk)
            self.ws_cf = torch.empty(B.ssm_conv_scan_workspace_size(csh, w.d_conv, False),
                                     dtype=torch.uint8, device=dev)
            self.ws_cb = torch.empty(B.ssm_conv_scan_workspace_size(csh, w.d_conv, True),
                                     dtype=torch.uint8, device=dev)
            if not w.fwd_only:
                self.gf = dict(self.g, d_sx=self.d_sx, d_c=self.d_c, d_bias=None)
                del self.gf["d_x"]

    def stages(self):
        B, w, d = self.B, self.w, self.d
        if self.path == "fused":
            out = [("conv_scan_fwd", lambda: B.ssm_conv_scan_fwd(
                d["sx"], d["c"], d["dt"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                s0=d["s0"], chunk=w.chunk, ws=self.ws_cf, out=(self.y, self.st, self.ck)))]
            if not w.fwd_only:
                out.append(("conv_scan_bwd", lambda: B.ssm_conv_scan_bwd(
                    d["sx"], d["c"], d["dt"], d["A"], d["B"], d["C"], d["dy"], D=d["D"],
                    z=d["z"], s0=d["s0"], ckpt=self.ck, d_state_out=d["d_state_out"],
                    chunk=w.chunk, ws=self.ws_cb, out=self.gf)))
            return out
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


def host_cores() -> int:
    """Host cores this process may run on (the oracle's threads use all of them)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _f64(t):
    import numpy as np
    if t is None:
        return None
    return np.ascontiguousarray(t.detach().to("cpu").double().numpy())


def oracle_slices(w, inp, seqs, parts):
    """The first `seqs` sequences of a workload's inputs cut into independent slices for the
    oracle: every slice holds whole sequences and whole tokens of a subset of channels (heads
    in the scalar-A form), converted to float64 once, outside any timed region.  Channels are
    independent except for the sums of dB and dC over channels, which each slice forms over
    its own channels (the same work)."""
    H, P = w.n_head, w.head_dim
    step = max(1, -(-H // max(1, parts)))
    out = []
    for h0 in range(0, H, step):
        h1 = min(H, h0 + step)
        c0, c1 = h0 * P, h1 * P
        sl = {"H": h1 - h0}
        if w.d_conv:
            sl["sx"] = _f64(inp["sx"][:seqs, c0:c1])
            sl["c"] = _f64(inp["c"][c0:c1])
            sl["x"] = None
        else:
            sl["x"] = _f64(inp["x"][:seqs, :, h0:h1])
        sl["dt"] = _f64(inp["dt"][:seqs, :, h0:h1])
        sl["A"] = _f64(inp["A"][h0:h1])
        sl["B"] = _f64(inp["B"][:seqs])
        sl["C"] = _f64(inp["C"][:seqs])
        sl["D"] = _f64(inp["D"][c0:c1]) if inp.get("D") is not None else None
        sl["z"] = _f64(inp["z"][:seqs, :, h0:h1]) if inp.get("z") is not None else None
        sl["s0"] = _f64(inp["s0"][:seqs, h0:h1]) if inp.get("s0") is not None else None
        sl["dy"] = _f64(inp["dy"][:seqs, :, h0:h1])
        out.append(sl)
    return out


def oracle_run(w, slices, seqs, threads):
    """Runs the oracle's whole step -- conv fwd, scan fwd (checkpoints), scan bwd from the
    checkpoints, conv bwd -- over `slices` on `threads` host threads (the oracle's C calls
    release the GIL).  Returns (forward seconds, backward seconds), each a wall-clock time."""
    import concurrent.futures as cf
    import oracle

    def dims(sl):
        return oracle.ScanDims(seqs, w.n_tok, sl["H"], w.head_dim, w.d_state, n_group=w.n_group,
                               a_per_state=0 if w.scalar_a else 1, chunk=w.chunk)

    def fwd(sl):
        x = sl["x"]
        if w.d_conv:
            x = oracle.conv_fwd(sl["sx"], sl["c"], None, silu=True)
            x = x.reshape(seqs, w.n_tok, sl["H"], w.head_dim)
        _, _, ck = oracle.scan_fwd(dims(sl), x=x, dt=sl["dt"], A=sl["A"], B=sl["B"], C=sl["C"],
                                   D=sl["D"], z=sl["z"], s0=sl["s0"])
        return x, ck

    def bwd(sl, x, ck):
        g = oracle.scan_bwd(dims(sl), x=x, dt=sl["dt"], A=sl["A"], B=sl["B"], C=sl["C"],
                            dy=sl["dy"], D=sl["D"], z=sl["z"], s0=sl["s0"], ckpt=ck)
        if w.d_conv:
            oracle.conv_bwd(sl["sx"], sl["c"], g["d_x"].reshape(seqs, w.n_tok, -1), silu=True)

    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        t0 = time.perf_counter()
        mid = list(ex.map(fwd, slices))
        t1 = time.perf_counter()
        bw_s = 0.0
        if not w.fwd_only:
            list(ex.map(lambda a: bwd(*a), [(sl, x, ck) for sl, (x, ck) in zip(slices, mid)]))
            bw_s = time.perf_counter() - t1
    return t1 - t0, bw_s


def oracle_seqs_for(w, inp, budget_cpu_s, cap=None):
    """How many whole sequences of the workload the oracle can run within `budget_cpu_s`
    seconds of CPU time (at least one), from a timed probe of one sequence x 2 channels."""
    probe = w.with_(n_head=2)
    f, b = oracle_run(probe, oracle_slices(probe, _probe_inputs(w, inp), 1, 1), 1, 1)
    per_seq = (f + b) * w.n_head / 2.0
    n = max(1, min(cap or w.n_seqs, int(budget_cpu_s / max(per_seq, 1e-9))))
    return n, per_seq


def _probe_inputs(w, inp):
    """The first two channels of the workload's inputs (all tokens, every sequence)."""
    H2, P = 2, w.head_dim
    out = dict(inp)
    for k in ("x", "z", "dy"):
        if inp.get(k) is not None:
            out[k] = inp[k][:, :, :H2]
    out["dt"] = inp["dt"][:, :, :H2]
    out["A"] = inp["A"][:H2]
    if inp.get("D") is not None:
        out["D"] = inp["D"][:H2 * P]
    if inp.get("c") is not None:
        out["c"] = inp["c"][:H2 * P]
    if inp.get("s0") is not None:
        out["s0"] = inp["s0"][:, :H2]
    return out


def oracle_baseline(w, inp, cores, budget_cpu_s):
    """The oracle on `cores` host threads over whole sequences of the workload (all of them if
    they fit the CPU-time budget), forward and backward timed separately."""
    seqs, _ = oracle_seqs_for(w, inp, budget_cpu_s)
    slices = oracle_slices(w, inp, seqs, 4 * cores if cores > 1 else 1)
    f, b = oracle_run(w, slices, seqs, cores)
    tok = seqs * w.n_tok
    rec = {"value": tok / (f + b), "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "fwd_s": f, "bwd_s": b, "fwd_tokens_s": tok / f,
           "sample": (f"{seqs} of {w.n_seqs} sequences x {w.n_tok} tokens x all {w.channels} "
                      f"channels of {w.name}: conv fwd + scan fwd (forward), scan bwd from the "
                      f"checkpoints + conv bwd (backward); f64 oracle on {cores} host threads "
                      f"over channel slices; inputs converted to f64 before timing")}
    if not w.fwd_only:
        rec["bwd_tokens_s"] = tok / b
    return rec


def cpu_baseline(w, inp, budget_cpu_s=30.0):
    """The oracle timed on all host cores on the bench's workload (whole sequences, all of them
    when they fit the budget), plus single-thread numbers on the two small configurations."""
    cores = host_cores()
    rec = oracle_baseline(w, inp, cores, budget_cpu_s)
    single = {}
    for small in WORKLOADS[:2]:
        si = make_inputs(small)
        r = oracle_baseline(small, si, 1, budget_cpu_s=1e9)
        single[small.name] = {k: r[k] for k in ("value", "fwd_s", "bwd_s") if k in r}
    rec["single_thread"] = single
    return rec


def run_reference(args, w):
    """The reference arm: the oracle, on all host cores, timed on whole sequences of the
    workload; each step runs the same sample, sized so that warm-up and timed steps end within
    about two minutes.  The line's value and ms_per_step are those of the steps it timed."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = make_inputs(w, grad_seed_state=False)
    cores = host_cores()
    budget_cpu = 120.0 * cores / max(1, args.steps + args.warmup)
    seqs, _ = oracle_seqs_for(w, inp, budget_cpu)
    slices = oracle_slices(w, inp, seqs, 4 * cores if cores > 1 else 1)
    for _ in range(args.warmup):
        oracle_run(w, slices, seqs, cores)
    times = [sum(oracle_run(w, slices, seqs, cores)) for _ in range(args.steps)]
    t_mean = sum(times) / len(times)
    value = seqs * w.n_tok / t_mean
    sample = (f"each step: {seqs} of {w.n_seqs} sequences x {w.n_tok} tokens x all "
              f"{w.channels} channels, full step (conv fwd, scan fwd, scan bwd, conv bwd), f64 "
              f"oracle on {cores} host threads; value and ms_per_step are of these steps")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * t_mean, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def stage_record(w, stage_ms, peaks) -> dict:
    """Per-stage time, achieved algorithmic GB/s and its fraction of the measured copy peak and
    of the 8 TB/s spec, for one workload."""
    ab = alg_bytes(w)
    tokens = w.n_seqs * w.n_tok
    gbs = {k: ab[k] * tokens / (stage_ms[k] * 1e-3) / 1e9 for k in stage_ms}
    return {"stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
            "stage_hbm_gbs": {k: round(v, 1) for k, v in gbs.items()},
            "stage_frac_of_measured": {k: round(v / peaks["hbm_gbs"], 4) for k, v in gbs.items()},
            "stage_frac_of_8tbs": {k: round(v / SPEC_HBM_GBS, 4) for k, v in gbs.items()}}


def roofline_of(w, stage_ms, peaks, peak_src, sms, mhz) -> dict:
    """Roofline of the dominant stage: algorithmic bytes per launch over its mean CUDA-event
    time against the measured HBM copy peak.  The ALU view (the method's own FP32 flops against
    the SMs' FP32 lanes at the sampled clock) rides along as a secondary field."""
    ab = alg_bytes(w)
    tokens = w.n_seqs * w.n_tok
    dom = max(stage_ms, key=stage_ms.get)
    dom_bytes = ab[dom] * tokens
    achieved = dom_bytes / (stage_ms[dom] * 1e-3) / 1e9
    traffic, traffic_kernel = captured_traffic(dom)
    roof = {"kernel": f"ssm_{dom}", "bound": "hbm", "achieved": achieved,
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "peak_source": peak_src, "traffic": traffic, "traffic_kernel": traffic_kernel,
            "algorithmic_bytes_per_launch": dom_bytes,
            "algorithmic_bytes_per_token": ab[dom]}
    if dom in SCAN_FLOPS:
        elems = tokens * w.channels * w.d_state
        flops = (SCAN_FLOPS_SCALAR_A if w.scalar_a else SCAN_FLOPS)[dom] * elems
        fp32_peak = sms * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
        ach_tf = flops / (stage_ms[dom] * 1e-3) / 1e12
        roof["alu"] = {"achieved": ach_tf, "peak": fp32_peak, "unit": "TFLOP/s",
                       "frac": ach_tf / fp32_peak, "algorithmic_flops_per_launch": flops,
                       "peak_source": f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 "
                                      f"x {mhz:.0f} MHz (sampled)"}
    return roof


def measure_target(w, dev, flush, steps, warmup, peaks, with_oracle, path="split") -> dict:
    """Stage times of another workload (or of the other path) on this GPU (device-timed as the
    main line, L2 flushed before every step), with its own clock record and, optionally, its
    oracle baseline."""
    inp = make_inputs(w, grad_seed_state=False)
    step = Step(w, dev, inp, path)
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t0 = time.time()
    total, per_stage, launches = time_device(step, steps, warmup, flush)
    t1 = time.time()
    clocks = sampler.stop(t0, t1)
    ms = sum(total) / len(total)
    stage_ms = {k: sum(v) / len(v) for k, v in per_stage.items()}
    rec = {"value": w.n_seqs * w.n_tok / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
           "path": step.path, "steps": steps, "warmup": warmup,
           **stage_record(w, stage_ms, peaks),
           "gpu_launches": int(launches), "clocks": clocks}
    del step
    if with_oracle:
        rec["cpu_baseline"] = oracle_baseline(w, inp, host_cores(), budget_cpu_s=30.0)
    return rec


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
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the second target configuration's and the other path's sub-records")
    ap.add_argument("--backward", action="store_true",
                    help="run the backward too on a forward-only workload (the Mamba-2 form)")
    ap.add_argument("--path", default="split", choices=["split", "fused"],
                    help="split: conv fwd, scan fwd, scan bwd, conv bwd as four calls; fused: "
                         "the conv1d+scan calls (x not kept between forward and backward)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    w = WORKLOADS[args.config] if args.config is not None else workload(args.workload)
    if args.backward and w.fwd_only:
        w = w.with_(fwd_only=False)
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
    step = Step(w, dev, inp, args.path)
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
    e2e_ms, h2d, d2h = time_e2e((step, Step(w, dev, inp, args.path)), e2e_steps, 2)
    e2e_ms = reduce_max(e2e_ms, dist, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    tokens = w.n_seqs * w.n_tok
    value = job_throughput(tokens, world, ms)
    peaks, peak_src = _measured_peaks()
    stage_ms = {k: sum(v) / len(v) for k, v in per_stage.items()}
    props = torch.cuda.get_device_properties(dev)
    mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz") or 2070.0
    roofline = roofline_of(w, stage_ms, peaks, peak_src, props.multi_processor_count, mhz)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.io == "bf16" else "f32", "data": "synthetic",
        "config": config_of(w, world), "path": step.path,
        **stage_record(w, stage_ms, peaks),
        "roofline": roofline,
        "gpu_launches": int(launches),
        "clocks": clocks,
        "e2e": {"value": job_throughput(tokens, world, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "pipelined": "2 buffer sets, copies of steps i+1 / i-1 overlap step i; inputs and results each one packed copy",
                "serial_ms_per_step": serial_ms},
    }
    if world == 1 and not args.no_targets and w.name in TARGET_WORKLOADS:
        line["targets"] = {w.name: {k: line[k] for k in ("stage_ms", "stage_hbm_gbs",
                                                         "stage_frac_of_measured",
                                                         "stage_frac_of_8tbs")}}
        for name in TARGET_WORKLOADS:
            if name != w.name:
                line["targets"][name] = measure_target(workload(name), dev, flush,
                                                       min(args.steps, 50), args.warmup,
                                                       peaks, not args.no_cpu_baseline)
    if world == 1 and not args.no_targets and w.d_conv and not w.fwd_only:
        other = "fused" if step.path == "split" else "split"
        line["other_path"] = measure_target(w, dev, flush, min(args.steps, 50), args.warmup,
                                            peaks, False, other)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, inp)
    print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
