"""Pins of the oracle's scan backward to things other than itself.

- the hand-worked example (tests/golden/scan_hand_l3_n1.json);
- central differences at eps = 1e-3 on ggmlR's tiny gradcheck shape (d_state 3, head_dim 2,
  n_head 2, 3 tokens, scalar A = -U(0.2, 1), dt ~ U(-1, 1), loss = <packed result, w>: test
  "ssm_scan gradients match a numeric gradient"), and on a Mamba-1 shape with gate, D,
  softplus dt and a dt bias;
- torch autograd in float64 through an independent torch implementation of the forward;
- zero upstream gradients give exactly zero gradients (gdn_backward.rs zero-grad test);
- the adjoint identity of the linear map (x, s0) -> (y, state_out) when D and z are absent;
- the checkpointed (TBPTT) backward equals the full-history one; duplicate ids accumulate.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import GRAD_ORDER, ScanDims
from bwd_ssm_conv_gb300.workloads import random_scan_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ev(v):
    return float(eval(v, {"ln2": math.log(2.0)})) if isinstance(v, str) else float(v)


def test_hand_worked_example_backward():
    with open(os.path.join(GOLDEN, "scan_hand_l3_n1.json")) as f:
        g = json.load(f)
    i = {k: np.array([_ev(v) for v in vals]) for k, vals in g["inputs"].items()}
    e = {k: np.array([_ev(v) for v in vals]) for k, vals in g["expected"].items()}
    dims = ScanDims(1, 3, 1, 1, 1, chunk=2)
    out = oracle.scan_bwd(dims, x=i["x"].reshape(1, 3, 1, 1), dt=i["dt"].reshape(1, 3, 1),
                          A=i["A"].reshape(1, 1), B=i["B"].reshape(1, 3, 1, 1),
                          C=i["C"].reshape(1, 3, 1, 1), D=i["D"], s0=i["s0"].reshape(1, 1, 1, 1),
                          dy=i["dy"].reshape(1, 3, 1, 1))
    for k in ("d_s0", "d_x", "d_B", "d_C", "d_dt", "d_A", "d_D"):
        np.testing.assert_allclose(out[k].ravel(), e[k], rtol=1e-13, atol=1e-13, err_msg=k)


def _loss_packed(dims, w_y, w_s, **kw):
    y, st, _ = oracle.scan_fwd(dims, want_ckpt=False, **kw)
    return float((y * w_y).sum() + (st * w_s).sum())


def _fd_check(dims, inputs, grads, names, eps=1e-3, rtol=2e-6, atol=1e-8, max_per=None):
    """Central differences of <packed forward, w> against the analytic gradients."""
    w_y, w_s = inputs.pop("_w_y"), inputs.pop("_w_s")
    for nm in names:
        base = np.array(inputs[nm], dtype=np.float64)
        g = grads["d_" + nm]
        idxs = list(np.ndindex(base.shape))
        if max_per is not None and len(idxs) > max_per:
            sel = np.random.default_rng(0).choice(len(idxs), max_per, replace=False)
            idxs = [idxs[j] for j in sel]
        for idx in idxs:
            hi, lo = base.copy(), base.copy()
            hi[idx] += eps
            lo[idx] -= eps
            f_hi = _loss_packed(dims, w_y, w_s, **{**inputs, nm: hi})
            f_lo = _loss_packed(dims, w_y, w_s, **{**inputs, nm: lo})
            num = (f_hi - f_lo) / (2 * eps)
            assert abs(num - g[idx]) <= atol + rtol * abs(num), (nm, idx, num, g[idx])


def test_fd_ggml_tiny_shape():
    rng = np.random.default_rng(21)
    N, P, H, L, ns = 3, 2, 2, 3, 1
    dims = ScanDims(ns, L, H, P, N, a_per_state=0, chunk=2)
    inp = dict(s0=rng.uniform(-1, 1, (ns, H, P, N)), x=rng.uniform(-1, 1, (ns, L, H, P)),
               dt=rng.uniform(-1, 1, (ns, L, H)), A=-rng.uniform(0.2, 1, H),
               B=rng.uniform(-1, 1, (ns, L, 1, N)), C=rng.uniform(-1, 1, (ns, L, 1, N)))
    w_y = rng.uniform(-1, 1, (ns, L, H, P))
    w_s = rng.uniform(-1, 1, (ns, H, P, N))
    grads = oracle.scan_bwd(dims, dy=w_y, d_state_out=w_s, **inp)
    _fd_check(dims, {**inp, "_w_y": w_y, "_w_s": w_s}, grads, ["s0", "x", "dt", "A", "B", "C"],
              rtol=1e-5, atol=1e-9)


def test_fd_mamba1_gate_D_softplus_bias():
    d = random_scan_inputs(2, 12, 3, 1, 4, seed=31, dt_raw=True)
    dims = ScanDims(2, 12, 3, 1, 4, chunk=5, dt_softplus=1)
    inp = {k: d[k].double().numpy() for k in ("x", "dt", "A", "B", "C", "D", "z", "s0")}
    inp["dt_bias"] = np.array([0.2, -0.4, 0.9])
    rng = np.random.default_rng(3)
    w_y = rng.normal(size=(2, 12, 3, 1))
    w_s = rng.normal(size=(2, 3, 1, 4))
    grads = oracle.scan_bwd(dims, dy=w_y, d_state_out=w_s, **inp)
    _fd_check(dims, {**inp, "_w_y": w_y, "_w_s": w_s}, grads,
              ["x", "dt", "A", "B", "C", "D", "z", "s0", "dt_bias"], rtol=1e-5, atol=1e-8,
              max_per=24)


def _torch_scan(x, dt, A, B, C, D, z, s0, dt_bias, a_per_state, softplus, G):
    """An independent float64 torch forward (vectorised over channels, loop over time)."""
    ns, L, H, P = x.shape
    N = B.shape[-1]
    delta = dt + dt_bias if (softplus and dt_bias is not None) else dt
    if softplus:
        delta = torch.nn.functional.softplus(delta)
    Ahn = A if a_per_state else A[:, None].expand(H, N)
    hidx = torch.arange(H) // (H // G)
    h = s0.clone() if s0 is not None else torch.zeros(ns, H, P, N, dtype=x.dtype)
    ys = []
    for t in range(L):
        dl = delta[:, t][:, :, None, None]                    # [ns, H, 1, 1]
        a = torch.exp(dl * Ahn[None, :, None, :])             # [ns, H, 1, N]
        Bt = B[:, t, hidx][:, :, None, :]                     # [ns, H, 1, N]
        Ct = C[:, t, hidx][:, :, None, :]
        h = a * h + dl * x[:, t][..., None] * Bt
        yp = (h * Ct).sum(-1)
        if D is not None:
            yp = yp + D.view(H, P) * x[:, t]
        if z is not None:
            yp = yp * torch.nn.functional.silu(z[:, t])
        ys.append(yp)
    return torch.stack(ys, 1), h


@pytest.mark.parametrize("case", ["mamba1", "mamba2_groups", "softplus"])
def test_backward_matches_torch_autograd(case):
    if case == "mamba1":
        ns, L, H, P, N, G, scal, sp = 2, 17, 4, 1, 5, 1, False, False
    elif case == "mamba2_groups":
        ns, L, H, P, N, G, scal, sp = 2, 9, 4, 3, 4, 2, True, False
    else:
        ns, L, H, P, N, G, scal, sp = 1, 11, 3, 2, 3, 1, False, True
    d = random_scan_inputs(ns, L, H, P, N, n_group=G, scalar_a=scal, seed=41, dt_raw=sp)
    t = {k: (v.double().clone().requires_grad_(True) if torch.is_tensor(v) else v)
         for k, v in d.items()}
    dt_bias = torch.tensor([0.3, -0.2, 0.5][:H], dtype=torch.float64,
                           requires_grad=True) if sp else None
    y, st = _torch_scan(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"], t["s0"],
                        dt_bias, not scal, sp, G)
    ((y * t["dy"]).sum() + (st * t["d_state_out"]).sum()).backward()
    dims = ScanDims(ns, L, H, P, N, n_group=G, a_per_state=0 if scal else 1, chunk=4,
                    dt_softplus=int(sp))
    o = oracle.scan_bwd(dims, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"], D=d["D"],
                        z=d["z"], s0=d["s0"], dy=d["dy"], d_state_out=d["d_state_out"],
                        dt_bias=None if dt_bias is None else dt_bias.detach())
    pairs = {"d_x": "x", "d_dt": "dt", "d_A": "A", "d_B": "B", "d_C": "C", "d_D": "D",
             "d_z": "z", "d_s0": "s0"}
    for gk, ik in pairs.items():
        np.testing.assert_allclose(o[gk], t[ik].grad.numpy(), rtol=1e-10, atol=1e-11, err_msg=gk)
    if sp:
        np.testing.assert_allclose(o["d_dt_bias"], dt_bias.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_softplus_threshold_matches_torch_autograd():
    """softplus is the identity above 20 (and its derivative 1 there), sigmoid-sloped below: dt
    biases near 20 put the pre-activations of two heads on both sides of the threshold, and the
    oracle's gradients equal torch's autograd of its own thresholded softplus (same convention)."""
    ns, L, H, P, N = 2, 9, 3, 1, 3
    d = random_scan_inputs(ns, L, H, P, N, seed=47, dt_raw=True)
    bias = torch.tensor([20.2, -0.3, 19.6], dtype=torch.float64)
    pre = d["dt"].double() + bias
    assert bool((pre > 20).any()) and bool((pre[..., [0, 2]] <= 20).any())
    t = {k: (v.double().clone().requires_grad_(True) if torch.is_tensor(v) else v)
         for k, v in d.items()}
    dt_bias = bias.clone().requires_grad_(True)
    y, st = _torch_scan(t["x"], t["dt"], t["A"], t["B"], t["C"], t["D"], t["z"], t["s0"],
                        dt_bias, True, True, 1)
    ((y * t["dy"]).sum() + (st * t["d_state_out"]).sum()).backward()
    dims = ScanDims(ns, L, H, P, N, chunk=4, dt_softplus=1)
    yo, so, _ = oracle.scan_fwd(dims, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"],
                                D=d["D"], z=d["z"], s0=d["s0"], dt_bias=bias.numpy())
    np.testing.assert_allclose(yo, y.detach().numpy(), rtol=1e-12, atol=1e-13)
    o = oracle.scan_bwd(dims, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"], D=d["D"],
                        z=d["z"], s0=d["s0"], dy=d["dy"], d_state_out=d["d_state_out"],
                        dt_bias=bias.numpy())
    np.testing.assert_allclose(o["d_dt"], t["dt"].grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(o["d_dt_bias"], dt_bias.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(o["d_x"], t["x"].grad.numpy(), rtol=1e-10, atol=1e-11)


def test_zero_upstream_gives_zero_gradients():
    d = random_scan_inputs(2, 10, 3, 2, 4, seed=5)
    dims = ScanDims(2, 10, 3, 2, 4, chunk=3)
    o = oracle.scan_bwd(dims, x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"], D=d["D"],
                        z=d["z"], s0=d["s0"], dy=np.zeros((2, 10, 3, 2)))
    for k in GRAD_ORDER:
        if o[k] is not None:
            assert not np.any(o[k]), k


def test_adjoint_identity_linear_map():
    # Without D and z, (x, s0) -> (y, state_out) is linear for fixed delta, B, C, so
    # <dy, y> + <dS, S> = <dx, x> + <ds0, s0> (the transpose of a linear map).
    d = random_scan_inputs(3, 25, 2, 3, 5, seed=6)
    dims = ScanDims(3, 25, 2, 3, 5, chunk=7)
    kw = dict(x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"], s0=d["s0"])
    y, st, _ = oracle.scan_fwd(dims, **kw)
    o = oracle.scan_bwd(dims, dy=d["dy"], d_state_out=d["d_state_out"], **kw)
    lhs = (y * d["dy"].double().numpy()).sum() + (st * d["d_state_out"].double().numpy()).sum()
    rhs = (o["d_x"] * d["x"].double().numpy()).sum() + (o["d_s0"] * d["s0"].double().numpy()).sum()
    assert abs(lhs - rhs) < 1e-11 * max(1.0, abs(lhs))


@pytest.mark.parametrize("chunk", [1, 4, 16, 50])
def test_checkpointed_equals_full_history(chunk):
    d = random_scan_inputs(2, 50, 3, 1, 4, seed=7)
    dims = ScanDims(2, 50, 3, 1, 4, chunk=chunk)
    kw = dict(x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"], D=d["D"], z=d["z"])
    _, _, ck = oracle.scan_fwd(dims, s0=d["s0"], **kw)
    full = oracle.scan_bwd(dims, s0=d["s0"], dy=d["dy"], d_state_out=d["d_state_out"], **kw)
    rec = oracle.scan_bwd(dims, ckpt=ck, dy=d["dy"], d_state_out=d["d_state_out"], **kw)
    for k in GRAD_ORDER:
        if full[k] is not None:
            np.testing.assert_array_equal(rec[k], full[k], err_msg=k)


def test_duplicate_ids_accumulate_and_unused_rows_are_zero():
    d = random_scan_inputs(3, 6, 2, 1, 3, seed=8)
    rows = np.random.default_rng(1).normal(size=(4, 2, 1, 3))
    ids = np.array([2, 0, 2], dtype=np.int32)
    kw = dict(x=d["x"], dt=d["dt"], A=d["A"], B=d["B"], C=d["C"], D=d["D"], z=d["z"],
              dy=d["dy"], d_state_out=d["d_state_out"])
    o = oracle.scan_bwd(ScanDims(3, 6, 2, 1, 3, state_rows=4), s0=rows, ids=ids, **kw)
    o_plain = oracle.scan_bwd(ScanDims(3, 6, 2, 1, 3), s0=rows[ids], **kw)
    np.testing.assert_array_equal(o["d_s0"][1], 0)
    np.testing.assert_array_equal(o["d_s0"][3], 0)
    np.testing.assert_allclose(o["d_s0"][0], o_plain["d_s0"][1], rtol=1e-15)
    np.testing.assert_allclose(o["d_s0"][2], o_plain["d_s0"][0] + o_plain["d_s0"][2], rtol=1e-14)
    np.testing.assert_array_equal(o["d_x"], o_plain["d_x"])
