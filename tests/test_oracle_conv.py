"""Pins of the oracle's conv1d (+bias, +SiLU) forward and backward to things other than itself.

- numpy.correlate per channel (a library routine; a flipped tap order would fail it);
- K = 1 with a unit weight reduces the op to a transpose;
- torch.nn.functional.conv1d + autograd in float64 (library) for the forward with bias/SiLU
  and for every gradient;
- ggmlR's closed form for loss = sum(out) (test "an ssm_conv node differentiates inside a
  backward graph"): d_c[k] = sum_t sx[t+k], and its mirror d_sx[i] = sum_{k: 0<=i-k<L} c[k];
- central differences at eps = 1e-3 (test "ssm_conv gradients match a numeric gradient").
"""
import numpy as np
import pytest
import torch

import oracle
from bwd_ssm_conv_gb300.workloads import random_conv_inputs


def _torch_conv(sx, c, bias, silu):
    # depthwise correlation: groups = channels, weight [D, 1, K]
    d = sx.shape[1]
    out = torch.nn.functional.conv1d(sx, c.view(d, 1, -1), bias=bias, groups=d)  # [n_s, D, L]
    if silu:
        out = torch.nn.functional.silu(out)
    return out.transpose(1, 2)  # [n_s, L, D]


@pytest.mark.parametrize("K", [1, 2, 3, 4, 7])
def test_conv_fwd_equals_numpy_correlate(K):
    inp = random_conv_inputs(2, 5, 9, K, seed=K)
    sx, c = inp["sx"].double().numpy(), inp["c"].double().numpy()
    out = oracle.conv_fwd(sx, c, silu=False)
    for b in range(2):
        for d in range(5):
            ref = np.correlate(sx[b, d], c[d], mode="valid")
            np.testing.assert_allclose(out[b, :, d], ref, rtol=0, atol=1e-13)


def test_conv_k1_unit_weight_is_transpose():
    inp = random_conv_inputs(3, 4, 11, 1, seed=3)
    sx = inp["sx"].double().numpy()
    out = oracle.conv_fwd(sx, np.ones((4, 1)), silu=False)
    np.testing.assert_array_equal(out, sx.transpose(0, 2, 1))


@pytest.mark.parametrize("silu,bias", [(True, False), (True, True), (False, True)])
def test_conv_fwd_matches_torch_conv1d(silu, bias):
    inp = random_conv_inputs(2, 6, 13, 4, bias=bias, seed=5)
    sx, c = inp["sx"].double(), inp["c"].double()
    bv = inp["bias"].double() if bias else None
    out = oracle.conv_fwd(sx, c, bv, silu=silu)
    ref = _torch_conv(sx, c, bv, silu).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-13, atol=1e-13)


def test_conv_state_out_is_last_columns():
    inp = random_conv_inputs(2, 3, 6, 4, seed=8)
    sx = inp["sx"].double().numpy()
    _, st = oracle.conv_fwd(sx, inp["c"], want_state=True)
    np.testing.assert_array_equal(st, sx[:, :, -3:])


@pytest.mark.parametrize("silu,bias", [(True, True), (False, False), (True, False)])
def test_conv_bwd_matches_torch_autograd(silu, bias):
    inp = random_conv_inputs(2, 5, 10, 4, bias=bias, seed=11)
    sx = inp["sx"].double().requires_grad_(True)
    c = inp["c"].double().requires_grad_(True)
    bv = inp["bias"].double().requires_grad_(True) if bias else None
    g = inp["dout"].double()
    out = _torch_conv(sx, c, bv, silu)
    (out * g).sum().backward()
    d_sx, d_c, d_b = oracle.conv_bwd(sx.detach(), c.detach(), g,
                                     bias=None if bv is None else bv.detach(), silu=silu)
    np.testing.assert_allclose(d_sx, sx.grad.numpy(), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(d_c, c.grad.numpy(), rtol=1e-12, atol=1e-12)
    if bias:
        np.testing.assert_allclose(d_b, bv.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_conv_bwd_sum_loss_closed_form():
    # ggmlR: with loss = sum(output) every upstream gradient is 1, so d_c[k] is the sum of
    # the sx values that tap k reads; by the same token d_sx[i] sums the taps that read i.
    K, L = 3, 4
    inp = random_conv_inputs(1, 2, L, K, seed=5)
    sx, c = inp["sx"].double().numpy(), inp["c"].double().numpy()
    d_sx, d_c, d_b = oracle.conv_bwd(sx, c, np.ones((1, L, 2)), silu=False)
    for d in range(2):
        for k in range(K):
            assert abs(d_c[d, k] - sx[0, d, k:k + L].sum()) < 1e-14
        for i in range(L + K - 1):
            ref = sum(c[d, k] for k in range(K) if 0 <= i - k < L)
            assert abs(d_sx[0, d, i] - ref) < 1e-14
    np.testing.assert_allclose(d_b, [L, L])


def test_conv_bwd_central_difference():
    # ggmlR "ssm_conv gradients match a numeric gradient": eps = 1e-3 on <out, g>
    inp = random_conv_inputs(2, 2, 4, 3, bias=True, seed=11)
    sx, c, bv = (inp[k].double().numpy() for k in ("sx", "c", "bias"))
    g = inp["dout"].double().numpy()
    d_sx, d_c, d_b = oracle.conv_bwd(sx, c, g, bias=bv, silu=True)

    def f(sx_, c_, b_):
        return float((oracle.conv_fwd(sx_, c_, b_, silu=True) * g).sum())

    eps = 1e-3
    for arr, grad, which in ((sx, d_sx, 0), (c, d_c, 1), (bv, d_b, 2)):
        for idx in np.ndindex(arr.shape):
            hi, lo = arr.copy(), arr.copy()
            hi[idx] += eps
            lo[idx] -= eps
            args_hi = [sx, c, bv]
            args_lo = [sx, c, bv]
            args_hi[which], args_lo[which] = hi, lo
            num = (f(*args_hi) - f(*args_lo)) / (2 * eps)
            assert abs(num - grad[idx]) < 1e-6 * max(1.0, abs(num)), (which, idx, num, grad[idx])
