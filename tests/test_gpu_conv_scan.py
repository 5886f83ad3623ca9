"""GPU parity of the conv1d(+bias, SiLU) -> selective scan path in one call (ssm_conv_scan_fwd,
ssm_conv_scan_bwd) against the oracle's chain: the conv, x rounded to the I/O type as the conv
would store it, the scan; and backward the scan's gradient followed by the conv's.

Backward, dL/dx passes between the scan's backward and the conv's in the I/O type (as between
ssm_scan_bwd and ssm_conv_bwd).  d_sx sums a few products of dL/dx and the weights and nearly
cancels in places, so one bf16 ulp of dL/dx moves it by more than the 2e-2 gate near zero (the
oracle's own d_sx from its rounded dL/dx differs from its exact one by 0.4 in the floored
metric).  The conv stage is therefore checked against the oracle's conv backward fed with the
dL/dx the GPU passes on (ssm_scan_bwd's output on the same inputs: the fused call runs the same
kernels), and the scan's gradients against the oracle's scan backward.

Shapes take the fused forward kernel (d_state 16, d_inner a multiple of 32, d_conv <= 4, tiles
of 16 tokens) or its fallback (x computed into the workspace): d_inner 40, d_state 8, d_conv 5.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import make_inputs, random_conv_inputs, random_scan_inputs, workload
from gpu_util import assert_close, nan_like, tol

pytestmark = pytest.mark.gpu

# name, (n_s, L, d_inner, d_state, d_conv), io, chunk, bias, silu, softplus
CASES = [
    ("fused_bf16", (2, 130, 64, 16, 4), "bf16", 32, True, True, False),
    ("fused_f32_k3_softplus", (1, 300, 96, 16, 3), "f32", 64, False, True, True),
    ("fused_bf16_k1_nosilu", (2, 64, 32, 16, 1), "bf16", 16, True, False, False),
    ("fused_bf16_k2_ragged", (3, 77, 64, 16, 2), "bf16", 48, True, True, False),
    ("fallback_channels40", (3, 77, 40, 16, 4), "bf16", 16, True, True, False),
    ("fallback_state8", (2, 50, 64, 8, 4), "bf16", 16, False, True, False),
    ("fallback_k5", (2, 90, 64, 16, 5), "f32", 32, True, True, False),
]


def _inputs(shape, io, bias, softplus, seed):
    n_s, L, d, N, K = shape
    cv = random_conv_inputs(n_s, d, L, K, io=io, bias=bias, seed=seed)
    sc = random_scan_inputs(n_s, L, d, 1, N, io=io, seed=seed + 1, dt_raw=softplus)
    inp = {"sx": cv["sx"], "c": cv["c"], "bias": cv["bias"]}
    for k in ("dt", "A", "B", "C", "D", "z", "s0", "dy", "d_state_out"):
        inp[k] = sc[k]
    inp["dt_bias"] = torch.linspace(-0.5, 0.5, d).float() if softplus else None
    return inp


def _x_ref(inp, silu):
    """The conv output as ssm_conv_fwd stores it (rounded to the I/O type), [n_s][L][d][1]."""
    x = oracle.conv_fwd(inp["sx"], inp["c"], inp["bias"], silu=silu)
    io = inp["sx"].dtype
    return torch.as_tensor(x).to(io).double().numpy()[..., None]


def _dims(inp, chunk, softplus):
    n_s, d, _ = inp["sx"].shape
    L = inp["dt"].shape[1]
    return oracle.ScanDims(n_s, L, d, 1, inp["B"].shape[3], chunk=chunk, dt_softplus=int(softplus))


def _gpu(inp):
    return {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_conv_scan_forward_parity(case):
    name, shape, io, chunk, bias, silu, softplus = case
    inp = _inputs(shape, io, bias, softplus, zlib.crc32(name.encode()) % 1000)
    d = _gpu(inp)
    n_s, L, dch, N, K = shape
    nch = (L + chunk - 1) // chunk
    out = (nan_like(d["sx"], (n_s, L, dch, 1)), nan_like(None, (n_s, dch, 1, N), torch.float32),
           nan_like(None, (n_s, nch, dch, 1, N), torch.float32))
    y, st, ck = binding.ssm_conv_scan_fwd(d["sx"], d["c"], d["dt"], d["A"], d["B"], d["C"],
                                          bias=d["bias"], silu=silu, D=d["D"], z=d["z"],
                                          dt_bias=d["dt_bias"], s0=d["s0"], chunk=chunk,
                                          softplus=softplus, out=out)
    x = _x_ref(inp, silu)
    yo, so, co = oracle.scan_fwd(_dims(inp, chunk, softplus), x=x, dt=inp["dt"], A=inp["A"],
                                 B=inp["B"], C=inp["C"], D=inp["D"], z=inp["z"],
                                 dt_bias=inp["dt_bias"], s0=inp["s0"])
    t = tol(io, grad=False)
    assert_close("y", y, yo, t)
    assert_close("state_out", st, so, t)
    assert_close("ckpt", ck, co, t)


@pytest.mark.parametrize("case", CASES[:2], ids=[c[0] for c in CASES[:2]])
def test_conv_scan_forward_equals_separate_calls(case):
    name, shape, io, chunk, bias, silu, softplus = case
    inp = _inputs(shape, io, bias, softplus, 7)
    d = _gpu(inp)
    n_s, L, dch, N, K = shape
    y, st, ck = binding.ssm_conv_scan_fwd(d["sx"], d["c"], d["dt"], d["A"], d["B"], d["C"],
                                          bias=d["bias"], silu=silu, D=d["D"], z=d["z"],
                                          dt_bias=d["dt_bias"], s0=d["s0"], chunk=chunk,
                                          softplus=softplus)
    x = binding.ssm_conv_fwd(d["sx"], d["c"], d["bias"], silu=silu).view(n_s, L, dch, 1)
    y2, st2, ck2 = binding.ssm_scan_fwd(x, d["dt"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                        dt_bias=d["dt_bias"], s0=d["s0"], chunk=chunk,
                                        softplus=softplus)
    t = tol(io, grad=False)
    assert_close("y", y, y2.float().cpu().numpy(), t)
    assert_close("state_out", st, st2.cpu().numpy(), t)
    assert_close("ckpt", ck, ck2.cpu().numpy(), t)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_conv_scan_backward_parity(case):
    name, shape, io, chunk, bias, silu, softplus = case
    inp = _inputs(shape, io, bias, softplus, zlib.crc32(name.encode()) % 1000 + 3)
    d = _gpu(inp)
    n_s, L, dch, N, K = shape
    _, _, ck = binding.ssm_conv_scan_fwd(d["sx"], d["c"], d["dt"], d["A"], d["B"], d["C"],
                                         bias=d["bias"], silu=silu, D=d["D"], z=d["z"],
                                         dt_bias=d["dt_bias"], s0=d["s0"], chunk=chunk,
                                         softplus=softplus)
    f32 = torch.float32
    out = dict(d_s0=nan_like(d["s0"]), d_sx=nan_like(d["sx"]), d_c=nan_like(d["c"]),
               d_bias=nan_like(None, (dch,), f32) if bias else None, d_dt=nan_like(d["dt"]),
               d_A=nan_like(d["A"]), d_B=nan_like(d["B"]), d_C=nan_like(d["C"]),
               d_D=nan_like(d["D"]), d_z=nan_like(d["z"]),
               d_dt_bias=nan_like(d["dt_bias"]) if softplus else None)
    g = binding.ssm_conv_scan_bwd(d["sx"], d["c"], d["dt"], d["A"], d["B"], d["C"], d["dy"],
                                  bias=d["bias"], silu=silu, D=d["D"], z=d["z"],
                                  dt_bias=d["dt_bias"], s0=d["s0"], ckpt=ck,
                                  d_state_out=d["d_state_out"], chunk=chunk, softplus=softplus,
                                  out=out)
    x = _x_ref(inp, silu)
    o = oracle.scan_bwd(_dims(inp, chunk, softplus), x=x, dt=inp["dt"], A=inp["A"], B=inp["B"],
                        C=inp["C"], dy=inp["dy"], D=inp["D"], z=inp["z"], dt_bias=inp["dt_bias"],
                        s0=inp["s0"], d_state_out=inp["d_state_out"])
    # the dL/dx the conv stage receives
    xg = binding.ssm_conv_fwd(d["sx"], d["c"], d["bias"], silu=silu).view(n_s, L, dch, 1)
    gs = binding.ssm_scan_bwd(xg, d["dt"], d["A"], d["B"], d["C"], d["dy"], D=d["D"], z=d["z"],
                              dt_bias=d["dt_bias"], s0=d["s0"], ckpt=ck,
                              d_state_out=d["d_state_out"], chunk=chunk, softplus=softplus)
    r_sx, r_c, r_b = oracle.conv_bwd(inp["sx"], inp["c"], gs["d_x"].cpu().view(n_s, L, dch),
                                     bias=inp["bias"], silu=silu)
    t = tol(io, grad=True)
    assert_close("d_x (conv stage input)", gs["d_x"], o["d_x"], t)
    assert_close("d_sx", g["d_sx"], r_sx, t)
    assert_close("d_c", g["d_c"], r_c, t)
    if bias:
        assert_close("d_bias", g["d_bias"], r_b, t)
    for k in ("d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_s0", "d_dt_bias"):
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], t)
    assert binding.ssm_scan_status(g["_ws"]) == 0


@pytest.mark.parametrize("name", ["mamba1_layer_f32_b8_l1024_d512_n16",
                                  "mamba1_long_bf16_b1_l16384_d2048_n16",
                                  "mamba1_train_bf16_b16_l2048_d1536_n16"])
def test_conv_scan_full_size_sampled_channels(name):
    """The Mamba-1 workloads (d_inner 512 x 8 x 1024 fp32, 2048 x 1 x 16384 and 1536 x 16 x
    2048 bf16) at full size through the fused calls, in the launch configuration the benchmark
    uses; the oracle runs the sampled channels (each channel's conv and scan are independent of
    the others)."""
    w = workload(name)
    inp = make_inputs(w, grad_seed_state=True)
    d = _gpu(inp)
    y, st, ck = binding.ssm_conv_scan_fwd(d["sx"], d["c"], d["dt"], d["A"], d["B"], d["C"],
                                          D=d["D"], z=d["z"], chunk=w.chunk)
    D = w.channels
    idx = torch.tensor(sorted({0, 1, 31, 32, 127, D // 2, D - 2, D - 1}), dtype=torch.long)
    sub = {"sx": inp["sx"][:, idx], "c": inp["c"][idx], "bias": None, "dt": inp["dt"][:, :, idx],
           "A": inp["A"][idx], "B": inp["B"], "C": inp["C"], "D": inp["D"][idx],
           "z": inp["z"][:, :, idx], "s0": None}
    x = _x_ref(sub, True)
    yo, so, co = oracle.scan_fwd(_dims(sub, w.chunk, False), x=x, dt=sub["dt"], A=sub["A"],
                                 B=sub["B"], C=sub["C"], D=sub["D"], z=sub["z"])
    t = tol(w.io, grad=False)
    assert_close("y", y[:, :, idx], yo, t)
    assert_close("state_out", st[:, idx], so, t)
    assert_close("ckpt", ck[:, :, idx], co, t)
    g = binding.ssm_conv_scan_bwd(d["sx"], d["c"], d["dt"], d["A"], d["B"], d["C"], d["dy"],
                                  D=d["D"], z=d["z"], ckpt=ck, d_state_out=d["d_state_out"],
                                  chunk=w.chunk)
    dy = inp["dy"][:, :, idx]
    o = oracle.scan_bwd(_dims(sub, w.chunk, False), x=x, dt=sub["dt"], A=sub["A"], B=sub["B"],
                        C=sub["C"], dy=dy, D=sub["D"], z=sub["z"],
                        d_state_out=inp["d_state_out"][:, idx])
    # the dL/dx the conv stage receives (see the module docstring)
    xg = binding.ssm_conv_fwd(d["sx"], d["c"], None, silu=True).view(w.n_seqs, w.n_tok, D, 1)
    gs = binding.ssm_scan_bwd(xg, d["dt"], d["A"], d["B"], d["C"], d["dy"], D=d["D"], z=d["z"],
                              ckpt=ck, d_state_out=d["d_state_out"], chunk=w.chunk)
    r_sx, r_c, _ = oracle.conv_bwd(sub["sx"], sub["c"],
                                   gs["d_x"][:, :, idx].cpu().view(w.n_seqs, w.n_tok, len(idx)),
                                   silu=True)
    tg = tol(w.io, grad=True)
    assert_close("d_sx", g["d_sx"][:, idx], r_sx, tg)
    assert_close("d_c", g["d_c"][idx], r_c, tg)
    for k in ("d_dt", "d_z"):
        assert_close(k, g[k][:, :, idx], o[k], tg)
    assert_close("d_A", g["d_A"][idx], o["d_A"], tg)
    assert_close("d_D", g["d_D"][idx], o["d_D"], tg)
