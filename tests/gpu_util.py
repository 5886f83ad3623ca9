"""Helpers for the GPU parity tests: run the CUDA path and the oracle on the same inputs."""
import numpy as np
import torch

import oracle
from oracle import ScanDims
from bwd_ssm_conv_gb300 import binding
from conftest import max_rel_err

# Tolerances on the floored max relative error (fp32 I/O forward / gradients; bf16 I/O).
TOL_F32_FWD = 1e-4
TOL_F32_GRAD = 1e-3
TOL_BF16 = 2e-2


def tol(io, grad):
    if io == "bf16" or io == torch.bfloat16:
        return TOL_BF16
    return TOL_F32_GRAD if grad else TOL_F32_FWD


def cuda(d):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in d.items()}


def assert_close(name, got, ref, tolerance):
    g = got.detach().float().cpu().numpy() if torch.is_tensor(got) else np.asarray(got)
    err = max_rel_err(g, ref)
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    assert err <= tolerance, f"{name}: max rel err {err:.3e} > {tolerance:.1e}"
    return err


def scan_dims(inp, chunk, softplus=False, state_rows=0):
    ns, L, H, P = inp["x"].shape
    G, N = inp["B"].shape[2], inp["B"].shape[3]
    return ScanDims(ns, L, H, P, N, n_group=G, a_per_state=1 if inp["A"].dim() == 2 else 0,
                    state_rows=state_rows, chunk=chunk, dt_softplus=int(softplus))


def nan_like(t, shape=None, dtype=None):
    """A CUDA output buffer filled with NaN: an element the kernels never write stays NaN and
    fails the parity check (assert_close rejects non-finite values)."""
    return torch.full(tuple(shape if shape is not None else t.shape), float("nan"),
                      dtype=dtype or t.dtype, device="cuda")


def gpu_fwd(inp, chunk, softplus=False, ids=None, state_rows=0, want_ckpt=True, chunked=False):
    d = cuda(inp)
    ns, L, H, P = inp["x"].shape
    N = inp["B"].shape[3]
    nch = (L + chunk - 1) // chunk
    out = (nan_like(d["x"]), nan_like(None, (ns, H, P, N), torch.float32),
           nan_like(None, (ns, nch, H, P, N), torch.float32) if want_ckpt else None)
    return binding.ssm_scan_fwd(d["x"], d["dt"], d["A"], d["B"], d["C"], D=d.get("D"),
                                z=d.get("z"), dt_bias=d.get("dt_bias"), s0=d.get("s0"),
                                ids=None if ids is None else ids.cuda(), chunk=chunk,
                                softplus=softplus, want_ckpt=want_ckpt, state_rows=state_rows,
                                out=out, chunked=chunked)


def gpu_bwd(inp, chunk, ckpt=None, softplus=False, ids=None, state_rows=0, d_state_out=True,
            check_finite=False, debug_flags=0):
    d = cuda(inp)
    ns, L, H, P = inp["x"].shape
    N = inp["B"].shape[3]
    rows = state_rows if state_rows else ns
    f32 = torch.float32
    out = dict(d_s0=nan_like(None, (rows, H, P, N), f32), d_x=nan_like(d["x"]),
               d_dt=nan_like(d["dt"]), d_A=nan_like(d["A"]), d_B=nan_like(d["B"]),
               d_C=nan_like(d["C"]),
               d_D=nan_like(d["D"]) if d.get("D") is not None else None,
               d_z=nan_like(d["z"]) if d.get("z") is not None else None,
               d_dt_bias=(nan_like(d["dt_bias"]) if d.get("dt_bias") is not None and softplus
                          else None))
    return binding.ssm_scan_bwd(d["x"], d["dt"], d["A"], d["B"], d["C"], d["dy"], D=d.get("D"),
                                z=d.get("z"), dt_bias=d.get("dt_bias"), s0=d.get("s0"),
                                ids=None if ids is None else ids.cuda(), ckpt=ckpt,
                                d_state_out=d.get("d_state_out") if d_state_out else None,
                                chunk=chunk, softplus=softplus, state_rows=state_rows, out=out,
                                check_finite=check_finite, debug_flags=debug_flags)


def oracle_fwd(inp, chunk, softplus=False, ids=None, state_rows=0):
    dims = scan_dims(inp, chunk, softplus, state_rows)
    return oracle.scan_fwd(dims, x=inp["x"], dt=inp["dt"], A=inp["A"], B=inp["B"], C=inp["C"],
                           D=inp.get("D"), z=inp.get("z"), dt_bias=inp.get("dt_bias"),
                           s0=inp.get("s0"), ids=ids)


def oracle_bwd(inp, chunk, softplus=False, ids=None, state_rows=0, d_state_out=True):
    dims = scan_dims(inp, chunk, softplus, state_rows)
    return oracle.scan_bwd(dims, x=inp["x"], dt=inp["dt"], A=inp["A"], B=inp["B"], C=inp["C"],
                           dy=inp["dy"], D=inp.get("D"), z=inp.get("z"),
                           dt_bias=inp.get("dt_bias"), s0=inp.get("s0"), ids=ids,
                           d_state_out=inp.get("d_state_out") if d_state_out else None)


def channel_subset(inp, idx):
    """The same problem restricted to Mamba-1 channels `idx` (head_dim 1, one group): every
    per-channel output of the subset equals the full problem's."""
    out = dict(inp)
    for k in ("x", "z", "dy"):
        if inp.get(k) is not None:
            out[k] = inp[k][:, :, idx]
    out["dt"] = inp["dt"][:, :, idx]
    out["A"] = inp["A"][idx]
    if inp.get("D") is not None:
        out["D"] = inp["D"][idx]
    if inp.get("dt_bias") is not None:
        out["dt_bias"] = inp["dt_bias"][idx]
    for k in ("s0", "d_state_out"):
        if inp.get(k) is not None:
            out[k] = inp[k][:, idx]
    return out
