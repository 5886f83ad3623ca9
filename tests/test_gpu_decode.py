"""Single-token decode: a loop that feeds one token at a time, carrying the conv state (the K-1
newest conv inputs) and the scan state between calls, gives the outputs of one call over the
whole sequence.  This is the step of infotheory's mamba1 runtime (forward_impl on one token with
its ring-buffer conv state and its recurrent state) and ggml's ssm_conv / ssm_scan with
n_seq_tokens = 1, run through the same entry points."""
import numpy as np
import pytest
import torch

import oracle
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


def _io(t, io):
    return t.to(torch.bfloat16).float() if io == "bf16" else t.float()


@pytest.mark.parametrize("io,P,N,G,scalar_a,softplus", [
    ("f32", 1, 16, 1, False, False),
    ("bf16", 1, 16, 1, False, True),
    ("f32", 4, 32, 2, True, True),     # Mamba-2 form with two groups
    ("bf16", 8, 128, 1, True, False),  # d_state 128: 32 threads per channel
    ("f32", 1, 256, 1, False, False),  # 8 states per thread
])
def test_fused_decode_step_matches_oracle(io, P, N, G, scalar_a, softplus):
    n_s, H, K, rows = 3, 8, 4, 5
    HP = H * P
    sc = random_scan_inputs(n_s, 1, H, P, N, n_group=G, io=io, scalar_a=scalar_a, has_z=True,
                            has_D=True, seed=21, dt_raw=softplus)
    g = torch.Generator().manual_seed(22)
    conv_state = _io(torch.randn(rows, HP, K - 1, generator=g), io)
    x_new = _io(torch.randn(n_s, HP, generator=g), io)
    c = (torch.rand(HP, K, generator=g) - 0.5).float()
    bias = (0.5 * torch.randn(HP, generator=g)).float()
    state = (0.5 * torch.randn(rows, H, P, N, generator=g)).float()
    dt_bias = torch.linspace(-0.5, 0.5, H).float() if softplus else None
    ids = torch.tensor([4, 0, 2], dtype=torch.int32)
    il = ids.long()

    # oracle: the conv over [conv_state | x_new], x stored in the io type, then one scan step
    sx = torch.cat([conv_state[il], x_new[:, :, None]], dim=2)
    xo = torch.as_tensor(np.asarray(oracle.conv_fwd(sx, c, bias, silu=True))).reshape(n_s, 1, H, P)
    dims = oracle.ScanDims(n_s, 1, H, P, N, n_group=G, a_per_state=0 if scalar_a else 1,
                           state_rows=rows, chunk=1, dt_softplus=int(softplus))
    yo, so, _ = oracle.scan_fwd(dims, x=_io(xo.float(), io), dt=sc["dt"], A=sc["A"], B=sc["B"],
                                C=sc["C"], D=sc["D"], z=sc["z"], dt_bias=dt_bias, s0=state,
                                ids=ids, want_ckpt=False)

    t_io = torch.bfloat16 if io == "bf16" else torch.float32
    cs_g = conv_state.to(t_io).cuda()
    st_g = state.cuda()
    y = binding.ssm_decode_step(
        x_new.to(t_io).view(n_s, H, P).cuda(), cs_g, c.cuda(), sc["dt"][:, 0].contiguous().cuda(),
        sc["A"].cuda(), sc["B"][:, 0].contiguous().cuda(), sc["C"][:, 0].contiguous().cuda(),
        st_g, bias=bias.cuda(), D=sc["D"].cuda(), z=sc["z"][:, 0].contiguous().cuda(),
        dt_bias=None if dt_bias is None else dt_bias.cuda(), ids=ids.cuda(), softplus=softplus,
        out=torch.full((n_s, H, P), float("nan"), dtype=t_io, device="cuda"))
    torch.cuda.synchronize()
    t = tol(io, grad=False)
    assert_close("y", y, np.asarray(yo).reshape(n_s, H, P), t)
    assert_close("state", st_g[il], np.asarray(so).reshape(n_s, H, P, N), t)
    untouched = [r for r in range(rows) if r not in ids.tolist()]
    assert torch.equal(st_g[untouched].cpu(), state[untouched])
    # the conv state rolls bit for bit; other rows stay
    rolled = torch.cat([conv_state[il][:, :, 1:], x_new[:, :, None]], dim=2).to(t_io)
    assert torch.equal(cs_g[il].cpu(), rolled)
    assert torch.equal(cs_g[untouched].cpu(), conv_state[untouched].to(t_io))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_fused_decode_loop_matches_full_sequence(io):
    n_s, d, L, K, N = 2, 64, 32, 4, 16
    cv = random_conv_inputs(n_s, d, L, K, io=io, bias=True, seed=31)
    sc = random_scan_inputs(n_s, L, d, 1, N, io=io, seed=32)
    sx, c, bias = cv["sx"].cuda(), cv["c"].cuda(), cv["bias"].cuda()
    dt, A, B, C = sc["dt"].cuda(), sc["A"].cuda(), sc["B"].cuda(), sc["C"].cuda()
    D, z, s0 = sc["D"].cuda(), sc["z"].cuda(), sc["s0"].cuda()
    x_full = binding.ssm_conv_fwd(sx, c, bias, silu=True)
    y_full, st_full, _ = binding.ssm_scan_fwd(x_full.view(n_s, L, d, 1), dt, A, B, C, D=D, z=z,
                                              s0=s0, chunk=16)
    conv_state = sx[:, :, :K - 1].contiguous()
    state = s0.clone()
    ys = []
    for t in range(L):
        ys.append(binding.ssm_decode_step(
            sx[:, :, K - 1 + t].contiguous().view(n_s, d, 1), conv_state, c, dt[:, t].contiguous(),
            A, B[:, t].contiguous(), C[:, t].contiguous(), state, bias=bias, D=D,
            z=z[:, t].contiguous()))
    torch.cuda.synchronize()
    y_dec = torch.stack(ys, dim=1)
    assert torch.equal(conv_state, sx[:, :, L:L + K - 1])
    t = tol(io, grad=False)
    assert_close("y", y_dec, y_full.float().cpu().numpy(), t)
    assert_close("state", state, st_full.float().cpu().numpy(), t)
