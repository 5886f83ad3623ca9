"""The device-side error paths, exercised without faulting the GPU.

* A cross-block wait that gives up: SSM_DEBUG_NO_WAIT makes every wait of a block on another
  block give up at once.  The persistent backward (resident blocks over (chain, chunk) units,
  each waiting for the adjoint that the unit of the next chunk publishes) must then record
  SSM_ERR_TIMEOUT, return promptly and leave the context usable.
* SSM_CHECK_FINITE: an infinite input must be reported as SSM_ERR_NONFINITE by the forward and
  the backward; without the flag, or with finite inputs, the status stays SSM_OK.
"""
import time

import pytest
import torch

from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import random_scan_inputs
from gpu_util import assert_close, gpu_bwd, gpu_fwd, oracle_bwd, tol

pytestmark = pytest.mark.gpu

# 24 sequences x 1024 channels = 768 chains of 32 channels: the persistent backward on a
# 152-SM GPU; 4 chunks of 16 tokens, so 3 of every chain's 4 units wait on a flag.
PERSIST = (24, 64, 1024, 1, 16, 1)


def _inp(shape, io, seed):
    ns, L, H, P, N, G = shape
    return random_scan_inputs(ns, L, H, P, N, n_group=G, io=io, seed=seed)


def test_flag_wait_gives_up_reports_timeout_and_leaves_the_context_usable():
    inp = _inp(PERSIST, "bf16", 51)
    _, _, ck = gpu_fwd(inp, 16)
    torch.cuda.synchronize()
    t0 = time.time()
    g = gpu_bwd(inp, 16, ckpt=ck, debug_flags=binding.SSM_DEBUG_NO_WAIT)
    status = binding.ssm_scan_status(g["_ws"])
    elapsed = time.time() - t0
    assert status == binding.SSM_ERR_TIMEOUT, binding.ssm_status_string(status)
    assert elapsed < 10.0, elapsed
    # the same call without the flag: the context still works and the results are right
    g = gpu_bwd(inp, 16, ckpt=ck)
    assert binding.ssm_scan_status(g["_ws"]) == binding.SSM_OK
    o = oracle_bwd(inp, 16)
    for k in ("d_x", "d_dt", "d_A", "d_B", "d_C", "d_D", "d_z", "d_s0"):
        assert_close(k, g[k], o[k], tol("bf16", grad=True))


@pytest.mark.parametrize("shape,io", [
    ((2, 70, 64, 1, 16, 1), "bf16"),   # TMA-staged kernels
    ((2, 70, 24, 1, 16, 1), "f32"),    # general kernels
])
def test_check_finite_reports_an_infinite_input(shape, io):
    inp = _inp(shape, io, 52)
    d = {k: (v.cuda() if torch.is_tensor(v) else v) for k, v in inp.items()}

    def fwd(x, check):
        _, _, _ = binding.ssm_scan_fwd(x, d["dt"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
                                       s0=d["s0"], chunk=32, check_finite=check, ws=ws_f)
        return binding.ssm_scan_status(ws_f)

    sh = binding.scan_shape(d["x"], d["dt"], d["A"], d["B"], d["s0"], 32)
    ws_f = torch.empty(binding.ssm_scan_workspace_size(sh, False), dtype=torch.uint8,
                       device="cuda")
    assert fwd(d["x"], True) == binding.SSM_OK
    x_inf = d["x"].clone()
    x_inf[1, 33, 5, 0] = float("inf")
    assert fwd(x_inf, False) == binding.SSM_OK
    assert fwd(x_inf, True) == binding.SSM_ERR_NONFINITE
    # the next call clears the word
    assert fwd(d["x"], True) == binding.SSM_OK

    _, _, ck = gpu_fwd(inp, 32)
    g = gpu_bwd(inp, 32, ckpt=ck, check_finite=True)
    assert binding.ssm_scan_status(g["_ws"]) == binding.SSM_OK
    bad = dict(inp)
    bad["dy"] = inp["dy"].clone()
    bad["dy"][0, 50, 7, 0] = float("inf")
    g = gpu_bwd(bad, 32, ckpt=ck, check_finite=True)
    assert binding.ssm_scan_status(g["_ws"]) == binding.SSM_ERR_NONFINITE
