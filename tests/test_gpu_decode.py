"""Single-token decode: a loop that feeds one token at a time, carrying the conv state (the K-1
newest conv inputs) and the scan state between calls, gives the outputs of one call over the
whole sequence.  This is the step of infotheory's mamba1 runtime (forward_impl on one token with
its ring-buffer conv state and its recurrent state) and ggml's ssm_conv / ssm_scan with
n_seq_tokens = 1, run through the same entry points."""
import pytest
import torch

from bwd_ssm_conv_gb300 import binding
from bwd_ssm_conv_gb300.workloads import random_conv_inputs, random_scan_inputs
from gpu_util import assert_close, tol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("io,N", [("f32", 16), ("bf16", 16), ("f32", 4)])
def test_decode_loop_matches_full_sequence(io, N):
    n_s, d, L, K = 2, 64, 40, 4
    cv = random_conv_inputs(n_s, d, L, K, io=io, bias=True, seed=11)
    sc = random_scan_inputs(n_s, L, d, 1, N, io=io, seed=12)
    sx, c, bias = cv["sx"].cuda(), cv["c"].cuda(), cv["bias"].cuda()
    dt, A, B, C = sc["dt"].cuda(), sc["A"].cuda(), sc["B"].cuda(), sc["C"].cuda()
    D, z, s0 = sc["D"].cuda(), sc["z"].cuda(), sc["s0"].cuda()

    # the whole sequence in one call of each
    x_full = binding.ssm_conv_fwd(sx, c, bias, silu=True)
    y_full, st_full, _ = binding.ssm_scan_fwd(x_full.view(n_s, L, d, 1), dt, A, B, C, D=D, z=z,
                                              s0=s0, chunk=16)

    # one token at a time
    conv_state = sx[:, :, :K - 1].contiguous()
    state = s0.clone()
    ys = []
    for t in range(L):
        sx_t = torch.cat([conv_state, sx[:, :, K - 1 + t:K + t]], dim=2).contiguous()
        x_t, conv_state = binding.ssm_conv_fwd(sx_t, c, bias, silu=True, want_state=True)
        y_t, state, _ = binding.ssm_scan_fwd(
            x_t.view(n_s, 1, d, 1), dt[:, t:t + 1].contiguous(), A, B[:, t:t + 1].contiguous(),
            C[:, t:t + 1].contiguous(), D=D, z=z[:, t:t + 1].contiguous(), s0=state, chunk=1,
            want_ckpt=False)
        ys.append(y_t)
    torch.cuda.synchronize()
    y_dec = torch.cat(ys, dim=1)

    # the conv state after the loop is the last K-1 inputs, bit for bit
    assert torch.equal(conv_state, sx[:, :, L:L + K - 1])
    t = tol(io, grad=False)
    assert_close("y", y_dec, y_full.float().cpu().numpy(), t)
    assert_close("state", state, st_full.float().cpu().numpy(), t)
