"""Backward of the Mamba-2 form on the head-tiled path (one A per head, head_dim a multiple of
32, d_state 128) with every optional input: gate z, skip D, softplus with dt_bias, groups,
time segments, a ragged last chunk; all gradients against the oracle."""
import pytest
import torch

from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import random_scan_inputs
from gpu_util import assert_close, gpu_bwd, gpu_fwd, oracle_bwd, tol

GRADS = ("d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_s0", "d_dt_bias")

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("io,shape,chunk,softplus", [
    ("f32", (2, 70, 4, 64, 128, 2), 16, False),
    ("bf16", (1, 90, 2, 96, 128, 1), 32, True),
])
def test_head_tiled_backward_with_gate_and_skip(io, shape, chunk, softplus):
    ns, L, H, P, N, G = shape
    inp = random_scan_inputs(ns, L, H, P, N, n_group=G, io=io, scalar_a=True, has_z=True,
                             has_D=True, seed=51, dt_raw=softplus)
    if softplus:
        inp["dt_bias"] = torch.linspace(-0.5, 0.5, H).float()
    _, _, ck = gpu_fwd(inp, chunk, softplus)
    g = gpu_bwd(inp, chunk, ckpt=ck, softplus=softplus)
    o = oracle_bwd(inp, chunk, softplus)
    t = tol(io, grad=True)
    for k in GRADS:
        if o.get(k) is not None and g.get(k) is not None:
            assert_close(k, g[k], o[k], t)
    assert binding.ssm_scan_status(g["_ws"]) == 0
